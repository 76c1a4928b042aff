// Switch load-balancing loss (S7) and its gradient (B7).
//
// The Ultimate MoE Training Handbook, §3.3 "Load balancing", part "Aux loss":
// the coefficient times the expert count times a sum over experts of each
// expert's share of the tokens times its mean router probability, i.e.
//     aux = coeff * E / (k * T^2) * sum_e counts[e] * sum_t P[t, e].
// P is the softmax of each token's logits over all E experts (for sigmoid
// scores, s / sum_e s). counts are integers and carry no gradient.
//
// Deterministic: a fixed partition of 64 tokens per CTA, fixed-order sums inside
// the CTA, per-CTA column sums written to scratch, and one CTA that adds them
// in block order (in fp64) and takes the dot with the counts.
#include "common.cuh"
#include "internal.h"

namespace moe {

constexpr int AUX_TOK = 64;  // tokens per CTA

static int64_t aux_blocks(int64_t T) { return (T + AUX_TOK - 1) / AUX_TOK; }

size_t aux_ws_bytes(const moe_cfg& cfg) {
  const size_t n = (size_t)aux_blocks(cfg.T) * (size_t)cfg.E * sizeof(float);
  return ((n + 255) & ~(size_t)255) + 256;
}

// P row of one token into p[EPL] (lane holds experts lane + 32 i); returns S for
// sigmoid (1 for softmax). Non-existent experts get 0.
template <int EPL>
__device__ __forceinline__ float token_probs(const float* __restrict__ row, int E, int score_fn,
                                             int lane, float (&p)[EPL], float (&s_out)[EPL]) {
  float l[EPL];
#pragma unroll
  for (int i = 0; i < EPL; ++i) {
    const int e = lane + 32 * i;
    l[i] = (e < E) ? row[e] : -INFINITY;
  }
  if (score_fn == MOE_SCORE_SOFTMAX) {
    float m = -INFINITY;
#pragma unroll
    for (int i = 0; i < EPL; ++i) m = fmaxf(m, l[i]);
    m = warp_max(m);
    float s = 0.f;
#pragma unroll
    for (int i = 0; i < EPL; ++i) {
      p[i] = (lane + 32 * i < E) ? expf(l[i] - m) : 0.f;
      s += p[i];
    }
    s = warp_sum(s);
    const float inv = 1.f / s;
#pragma unroll
    for (int i = 0; i < EPL; ++i) {
      p[i] *= inv;
      s_out[i] = 0.f;
    }
    return 1.f;
  }
  float s = 0.f;
#pragma unroll
  for (int i = 0; i < EPL; ++i) {
    s_out[i] = (lane + 32 * i < E) ? sigmoidf_acc(l[i]) : 0.f;
    s += s_out[i];
  }
  s = warp_sum(s);
  const float inv = 1.f / s;
#pragma unroll
  for (int i = 0; i < EPL; ++i) p[i] = s_out[i] * inv;
  return s;
}

template <int EPL>
__global__ void __launch_bounds__(256)
aux_partials(const float* __restrict__ logits, int64_t T, int E, int score_fn,
             float* __restrict__ part) {
  __shared__ float wsum[8][kMaxE];
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  float col[EPL];
#pragma unroll
  for (int i = 0; i < EPL; ++i) col[i] = 0.f;
  const int64_t t0 = (int64_t)blockIdx.x * AUX_TOK;
  for (int tl = warp; tl < AUX_TOK; tl += 8) {
    const int64_t t = t0 + tl;
    if (t >= T) break;
    float p[EPL], s[EPL];
    token_probs<EPL>(logits + t * E, E, score_fn, lane, p, s);
#pragma unroll
    for (int i = 0; i < EPL; ++i) col[i] += p[i];
  }
#pragma unroll
  for (int i = 0; i < EPL; ++i) {
    const int e = lane + 32 * i;
    if (e < E) wsum[warp][e] = col[i];
  }
  __syncthreads();
  for (int e = threadIdx.x; e < E; e += blockDim.x) {
    float v = 0.f;
#pragma unroll
    for (int w = 0; w < 8; ++w) v += wsum[w][e];
    part[(int64_t)blockIdx.x * E + e] = v;
  }
}

__global__ void __launch_bounds__(256)
aux_finalize(const float* __restrict__ part, int64_t nblk, const int32_t* __restrict__ counts,
             int64_t T, int E, int k, float coeff, float* __restrict__ aux) {
  __shared__ double term[kMaxE];
  const int e = threadIdx.x;
  if (e < E) {
    double col = 0.0;
    for (int64_t b = 0; b < nblk; ++b) col += (double)part[b * E + e];
    term[e] = col * (double)counts[e];
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    double acc = 0.0;
    for (int i = 0; i < E; ++i) acc += term[i];
    const double scale =
        (T > 0) ? (double)coeff * (double)E / ((double)k * (double)T * (double)T) : 0.0;
    *aux = (float)(acc * scale);
  }
}

template <int EPL>
__global__ void __launch_bounds__(256)
aux_bwd_kernel(const float* __restrict__ logits, const int32_t* __restrict__ counts, int64_t T,
               int E, int k, int score_fn, float g_scale, float* __restrict__ d_logits,
               int accumulate) {
  const int lane = threadIdx.x & 31;
  const int64_t nwarps = ((int64_t)gridDim.x * blockDim.x) >> 5;
  float dP[EPL];
#pragma unroll
  for (int i = 0; i < EPL; ++i) {
    const int e = lane + 32 * i;
    dP[i] = (e < E) ? g_scale * (float)counts[e] : 0.f;
  }
  for (int64_t t = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5; t < T; t += nwarps) {
    float p[EPL], s[EPL];
    const float S = token_probs<EPL>(logits + t * E, E, score_fn, lane, p, s);
    float dot = 0.f;
#pragma unroll
    for (int i = 0; i < EPL; ++i) dot += p[i] * dP[i];
    dot = warp_sum(dot);
#pragma unroll
    for (int i = 0; i < EPL; ++i) {
      const int e = lane + 32 * i;
      if (e < E) {
        float g;
        if (score_fn == MOE_SCORE_SOFTMAX) {
          g = p[i] * (dP[i] - dot);
        } else {
          g = (dP[i] - dot) / S * s[i] * (1.f - s[i]);
        }
        float* dst = d_logits + t * E + e;
        *dst = accumulate ? *dst + g : g;
      }
    }
  }
}

cudaError_t launch_aux_loss(const Ctx& c, const moe_cfg& cfg, const float* logits,
                            const int32_t* counts, float* aux, void* ws) {
  const int64_t nblk = aux_blocks(cfg.T);
  float* part = static_cast<float*>(ws);
  const int epl = (cfg.E + 31) / 32;
  if (nblk > 0) {
#define MOE_AUXP(N) \
  aux_partials<N><<<(unsigned)nblk, 256, 0, c.stream>>>(logits, cfg.T, cfg.E, cfg.score_fn, part)
    switch (epl) {
      case 1: MOE_AUXP(1); break;
      case 2: MOE_AUXP(2); break;
      case 3: case 4: MOE_AUXP(4); break;
      default: MOE_AUXP(8); break;
    }
#undef MOE_AUXP
  }
  aux_finalize<<<1, 256, 0, c.stream>>>(part, nblk, counts, cfg.T, cfg.E, cfg.k, cfg.aux_coeff,
                                        aux);
  note_launches(nblk > 0 ? 2 : 1);
  return cudaGetLastError();
}

cudaError_t launch_aux_loss_bwd(const Ctx& c, const moe_cfg& cfg, const float* logits,
                                const int32_t* counts, float g_aux, float* d_logits,
                                int accumulate) {
  if (cfg.T == 0) return cudaSuccess;
  const double Td = (double)cfg.T;
  const float g_scale =
      (float)((double)g_aux * (double)cfg.aux_coeff * (double)cfg.E / ((double)cfg.k * Td * Td));
  const int64_t blocks = (cfg.T + 7) / 8;
  const int64_t cap = (int64_t)c.sm_count * 8;
  const unsigned grid = (unsigned)(blocks < cap ? blocks : cap);
  const int epl = (cfg.E + 31) / 32;
#define MOE_AUXB(N)                                                                        \
  aux_bwd_kernel<N><<<grid, 256, 0, c.stream>>>(logits, counts, cfg.T, cfg.E, cfg.k,      \
                                                cfg.score_fn, g_scale, d_logits, accumulate)
  switch (epl) {
    case 1: MOE_AUXB(1); break;
    case 2: MOE_AUXB(2); break;
    case 3: case 4: MOE_AUXB(4); break;
    default: MOE_AUXB(8); break;
  }
#undef MOE_AUXB
  note_launches(1);
  return cudaGetLastError();
}

}  // namespace moe
