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

// P row of one token into p[EPL] (lane holds experts lane + 32 i): the softmax
// over all E, or s / sum_e s for the sigmoid-like scores (s_out = s, returns
// sum_e s; 1 for softmax). l_out receives the logits. Non-existent experts
// get 0.
template <int EPL>
__device__ __forceinline__ float token_probs(const float* __restrict__ row, int E, int score_fn,
                                             int lane, float (&p)[EPL], float (&s_out)[EPL],
                                             float (&l)[EPL]) {
#pragma unroll
  for (int i = 0; i < EPL; ++i) {
    const int e = lane + 32 * i;
    l[i] = (e < E) ? row[e] : -INFINITY;
  }
  if (score_fn == MOE_SCORE_SOFTMAX || score_fn == MOE_SCORE_SOFTMAX_PRE) {
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
    s_out[i] = (lane + 32 * i < E) ? bias_score(l[i], score_fn) : 0.f;
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
  pdl_wait();  // a dependent launch: inputs come from the kernels before
  __shared__ float wsum[8][kMaxE];
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  float col[EPL];
#pragma unroll
  for (int i = 0; i < EPL; ++i) col[i] = 0.f;
  const int64_t t0 = (int64_t)blockIdx.x * AUX_TOK;
  for (int tl = warp; tl < AUX_TOK; tl += 8) {
    const int64_t t = t0 + tl;
    if (t >= T) break;
    float p[EPL], s[EPL], l[EPL];
    token_probs<EPL>(logits + t * E, E, score_fn, lane, p, s, l);
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

// The same per-CTA column sums for few experts (E <= G <= 16): G lanes per
// token (lane e of a group holds expert e), so a warp takes 32 / G tokens at
// once instead of one with E of its 32 lanes busy; each warp's 8 tokens are
// loaded before any is reduced. Lane e adds its tokens' probabilities, the
// token slots of the warp add by a fixed butterfly, the warps in order
// (Mixtral-style sizes, T = 4096, E = 8: the aux-loss stage 18.4 -> 12.1 us).
template <int G>
__global__ void __launch_bounds__(256)
aux_partials_grouped(const float* __restrict__ logits, int64_t T, int E, int score_fn,
                     float* __restrict__ part) {
  pdl_wait();  // a dependent launch: inputs come from the kernels before
  static_assert(AUX_TOK == 8 * 8, "eight warps of eight tokens");
  constexpr int SLOTS = 32 / G, PASSES = 8 / SLOTS;
  __shared__ float wsum[8][G];
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int e = lane & (G - 1), slot = lane / G;
  const bool real = e < E;
  const bool soft = score_fn == MOE_SCORE_SOFTMAX || score_fn == MOE_SCORE_SOFTMAX_PRE;
  const int64_t tw = (int64_t)blockIdx.x * AUX_TOK + warp * 8;  // the warp's 8 tokens
  float l[PASSES];
#pragma unroll
  for (int q = 0; q < PASSES; ++q) {
    const int64_t t = tw + q * SLOTS + slot;
    l[q] = (real && t < T) ? logits[t * E + e] : -INFINITY;
  }
  float col = 0.f;
#pragma unroll
  for (int q = 0; q < PASSES; ++q) {
    const int64_t t = tw + q * SLOTS + slot;
    float p;
    if (soft) {
      float m = l[q];
#pragma unroll
      for (int o = G / 2; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o, G));
      p = real ? expf(l[q] - m) : 0.f;
    } else {
      p = real ? bias_score(l[q], score_fn) : 0.f;
    }
    float sum = p;
#pragma unroll
    for (int o = G / 2; o > 0; o >>= 1) sum += __shfl_xor_sync(0xffffffffu, sum, o, G);
    if (t < T) col += p * (1.f / sum);
  }
#pragma unroll
  for (int o = 16; o >= G; o >>= 1) col += __shfl_xor_sync(0xffffffffu, col, o);
  if (lane < G) wsum[warp][lane] = col;
  __syncthreads();
  for (int c = threadIdx.x; c < E; c += blockDim.x) {
    float v = 0.f;
#pragma unroll
    for (int w = 0; w < 8; ++w) v += wsum[w][c];
    part[(int64_t)blockIdx.x * E + c] = v;
  }
}

// 1024 threads: thread (j, e) sums the block partials b = j, j + J, j + 2J,
// ... of column e into a compensated fp32 pair (J = min(1024 / E, 32) lanes
// per column), the J pairs of a column are added in j order (TwoSum), the
// column total times the count is formed in fp64, and the E terms are added
// by a fixed pairwise tree: the same order on every run, and short dependent
// chains of cheap operations (fp64 is slow on this part).
__global__ void __launch_bounds__(1024)
aux_finalize(const float* __restrict__ part, int64_t nblk, const int32_t* __restrict__ counts,
             int64_t T, int E, int k, float coeff, float* __restrict__ aux) {
  pdl_wait();  // a dependent launch: inputs come from the kernels before
  __shared__ float colh[1024];
  __shared__ float coll[1024];
  __shared__ double term[kMaxE];
  int J = E > 0 ? 1024 / E : 1;
  J = J < 1 ? 1 : (J > 32 ? 32 : J);
  for (int q = threadIdx.x; q < J * E; q += blockDim.x) {
    const int j = q / E, e = q - j * E;
    float hi = 0.f, lo = 0.f;
#pragma unroll 4
    for (int64_t b = j; b < nblk; b += J) comp_add(hi, lo, part[b * E + e]);
    colh[q] = hi;
    coll[q] = lo;
  }
  __syncthreads();
  for (int e = threadIdx.x; e < E; e += blockDim.x) {
    float hi = colh[e], lo = coll[e];
    for (int j = 1; j < J; ++j) {
      float s, er;
      two_sum(hi, colh[j * E + e], s, er);
      hi = s;
      lo = __fadd_rn(__fadd_rn(lo, coll[j * E + e]), er);
    }
    term[e] = ((double)hi + (double)lo) * (double)counts[e];
  }
  __syncthreads();
  // pairwise tree over the E terms (E <= 256)
  for (int width = 1; width < E; width <<= 1) {
    for (int i = threadIdx.x * 2 * width; i + width < E; i += blockDim.x * 2 * width)
      term[i] += term[i + width];
    __syncthreads();
  }
  if (threadIdx.x == 0) {
    const double scale =
        (T > 0) ? (double)coeff * (double)E / ((double)k * (double)T * (double)T) : 0.0;
    *aux = (float)((E > 0 ? term[0] : 0.0) * scale);
  }
}

template <int EPL>
__global__ void __launch_bounds__(256)
aux_bwd_kernel(const float* __restrict__ logits, const int32_t* __restrict__ counts, int64_t T,
               int E, int k, int score_fn, float g_scale, float* __restrict__ d_logits,
               int accumulate) {
  pdl_wait();  // a dependent launch: inputs come from the kernels before
  const int lane = threadIdx.x & 31;
  const int64_t nwarps = ((int64_t)gridDim.x * blockDim.x) >> 5;
  float dP[EPL];
#pragma unroll
  for (int i = 0; i < EPL; ++i) {
    const int e = lane + 32 * i;
    dP[i] = (e < E) ? g_scale * (float)counts[e] : 0.f;
  }
  for (int64_t t = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5; t < T; t += nwarps) {
    float p[EPL], s[EPL], l[EPL];
    const float S = token_probs<EPL>(logits + t * E, E, score_fn, lane, p, s, l);
    float dot = 0.f;
#pragma unroll
    for (int i = 0; i < EPL; ++i) dot += p[i] * dP[i];
    dot = warp_sum(dot);
#pragma unroll
    for (int i = 0; i < EPL; ++i) {
      const int e = lane + 32 * i;
      if (e < E) {
        float g;
        if (score_fn == MOE_SCORE_SOFTMAX || score_fn == MOE_SCORE_SOFTMAX_PRE) {
          g = p[i] * (dP[i] - dot);
        } else {
          g = (dP[i] - dot) / S * bias_score_deriv(l[i], s[i], score_fn);
        }
        float* dst = d_logits + t * E + e;
        *dst = accumulate ? *dst + g : g;
      }
    }
  }
}

// ---------------------------------------------------------------- router z-loss
// Handbook §3.1 "Router scoring", part "Precision" (z_loss_func):
//   z = coeff * mean_t (logsumexp_t l)^2,  dz/dl[t, e] = coeff * 2 lse_t softmax(l_t)_e / T.
// Deterministic like the aux loss: 64 tokens per CTA, fixed-order sums, fp64
// partials added in block order by one thread.
constexpr int Z_TOK = 64;

size_t z_loss_ws_bytes(const moe_cfg& cfg) {
  const size_t n = (size_t)((cfg.T + Z_TOK - 1) / Z_TOK) * sizeof(double);
  return ((n + 255) & ~(size_t)255) + 256;
}

template <int EPL>
__device__ __forceinline__ float token_lse(const float* __restrict__ row, int E, int lane,
                                           float (&l)[EPL], float& m_out, float& sum_out) {
  float m = -INFINITY;
#pragma unroll
  for (int i = 0; i < EPL; ++i) {
    const int e = lane + 32 * i;
    l[i] = (e < E) ? row[e] : -INFINITY;
    m = fmaxf(m, l[i]);
  }
  m = warp_max(m);
  float sum = 0.f;
#pragma unroll
  for (int i = 0; i < EPL; ++i)
    if (lane + 32 * i < E) sum += expf(l[i] - m);
  sum = warp_sum(sum);
  m_out = m;
  sum_out = sum;
  return m + logf(sum);
}

template <int EPL>
__global__ void __launch_bounds__(256)
z_partials(const float* __restrict__ logits, int64_t T, int E, double* __restrict__ part) {
  __shared__ double wsum[8];
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  double acc = 0.0;
  const int64_t t0 = (int64_t)blockIdx.x * Z_TOK;
  for (int tl = warp; tl < Z_TOK; tl += 8) {
    const int64_t t = t0 + tl;
    if (t >= T) break;
    float l[EPL], m, sum;
    const float lse = token_lse<EPL>(logits + t * E, E, lane, l, m, sum);
    acc += (double)lse * (double)lse;
  }
  if (lane == 0) wsum[warp] = acc;
  __syncthreads();
  if (threadIdx.x == 0) {
    double v = 0.0;
    for (int w = 0; w < 8; ++w) v += wsum[w];
    part[blockIdx.x] = v;
  }
}

__global__ void z_finalize(const double* __restrict__ part, int64_t nblk, int64_t T, float coeff,
                           float* __restrict__ z) {
  if (threadIdx.x != 0 || blockIdx.x != 0) return;
  double v = 0.0;
#pragma unroll 8
  for (int64_t b = 0; b < nblk; ++b) v += part[b];
  *z = (T > 0) ? (float)((double)coeff * v / (double)T) : 0.f;
}

template <int EPL>
__global__ void __launch_bounds__(256)
z_bwd_kernel(const float* __restrict__ logits, int64_t T, int E, float g_scale,
             float* __restrict__ d_logits, int accumulate) {
  const int lane = threadIdx.x & 31;
  const int64_t nwarps = ((int64_t)gridDim.x * blockDim.x) >> 5;
  for (int64_t t = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5; t < T; t += nwarps) {
    float l[EPL], m, sum;
    const float lse = token_lse<EPL>(logits + t * E, E, lane, l, m, sum);
    const float f = g_scale * lse / sum;
#pragma unroll
    for (int i = 0; i < EPL; ++i) {
      const int e = lane + 32 * i;
      if (e < E) {
        const float g = f * expf(l[i] - m);
        float* dst = d_logits + t * E + e;
        *dst = accumulate ? *dst + g : g;
      }
    }
  }
}

#define MOE_BY_EPL(EPLV, MACRO) \
  switch (EPLV) {               \
    case 1: MACRO(1); break;    \
    case 2: MACRO(2); break;    \
    case 3: case 4: MACRO(4); break; \
    default: MACRO(8); break;   \
  }

cudaError_t launch_z_loss(const Ctx& c, const moe_cfg& cfg, const float* logits, float coeff,
                          float* z, void* ws) {
  const int64_t nblk = (cfg.T + Z_TOK - 1) / Z_TOK;
  double* part = static_cast<double*>(ws);
  const int epl = (cfg.E + 31) / 32;
  if (nblk > 0) {
#define MOE_ZP(N) z_partials<N><<<(unsigned)nblk, 256, 0, c.stream>>>(logits, cfg.T, cfg.E, part)
    MOE_BY_EPL(epl, MOE_ZP)
#undef MOE_ZP
  }
  z_finalize<<<1, 32, 0, c.stream>>>(part, nblk, cfg.T, coeff, z);
  note_launches(nblk > 0 ? 2 : 1);
  return cudaGetLastError();
}

cudaError_t launch_z_loss_bwd(const Ctx& c, const moe_cfg& cfg, const float* logits, float coeff,
                              float g_z, float* d_logits, int accumulate) {
  if (cfg.T == 0) return cudaSuccess;
  const float g_scale = (float)((double)g_z * (double)coeff * 2.0 / (double)cfg.T);
  const int64_t blocks = (cfg.T + 7) / 8;
  const int64_t cap = (int64_t)c.sm_count * 8;
  const unsigned grid = (unsigned)(blocks < cap ? blocks : cap);
  const int epl = (cfg.E + 31) / 32;
#define MOE_ZB(N)                                                                          \
  z_bwd_kernel<N><<<grid, 256, 0, c.stream>>>(logits, cfg.T, cfg.E, g_scale, d_logits, \
                                              accumulate)
  MOE_BY_EPL(epl, MOE_ZB)
#undef MOE_ZB
  note_launches(1);
  return cudaGetLastError();
}

// ---------------------------------------------------------------- sequence-wise aux loss
// Handbook §3.3 "Load balancing", part "Scope" (seq_aux_loss): the Switch loss
// of each sequence on its own (its counts, its probabilities, its length S),
// averaged over the B = T / S sequences:
//   (1/B) sum_b coeff * E / (k * S^2) * sum_e c[b, e] * sum_{t in b} P[t, e].
// Token t of sequence b, position s: t = b S + s (batch-major) or t = s B + b
// (sequence-major, the [seq, batch] order of Megatron's activations).
// A sequence is cut into `cps` chunks of up to `chunk` tokens; one CTA per
// chunk writes its column sums of P and its expert counts; the sums over
// chunks, experts and sequences then run in fixed order (deterministic).
struct SeqPlan {
  int64_t B, S, cps, chunk;
};

static SeqPlan seq_plan(const moe_cfg& cfg, int64_t S) {
  SeqPlan p;
  p.S = S;
  p.B = cfg.T / S;
  const int64_t max_cps = (S + 63) / 64;
  int64_t cps = (1024 + p.B - 1) / p.B;  // about 1024 CTAs in all
  if (cps > max_cps) cps = max_cps;
  if (cps < 1) cps = 1;
  p.cps = cps;
  p.chunk = (S + cps - 1) / cps;
  return p;
}

size_t seq_aux_ws_bytes(const moe_cfg& cfg, int64_t S) {
  if (S <= 0 || cfg.T % S != 0) return 0;
  const SeqPlan p = seq_plan(cfg, S);
  const size_t n = (size_t)(p.B * p.cps) * (size_t)cfg.E;
  const size_t a = ((n * sizeof(float) + 255) & ~(size_t)255);        // column sums
  const size_t b = ((n * sizeof(int32_t) + 255) & ~(size_t)255);      // counts
  const size_t c = (((size_t)p.B * sizeof(double) + 255) & ~(size_t)255);  // per-sequence losses
  const size_t d = (((size_t)p.B * cfg.E * sizeof(int32_t) + 255) & ~(size_t)255);  // counts per sequence
  return a + b + c + d + 256;
}

__device__ __forceinline__ int64_t seq_token(int64_t b, int64_t s, int64_t B, int64_t S,
                                             int seq_major) {
  return seq_major ? s * B + b : b * S + s;
}

// colsum may be NULL (counts only)
template <int EPL>
__global__ void __launch_bounds__(256)
seq_partials(const float* __restrict__ logits, const int32_t* __restrict__ idx, int E, int k,
             SeqPlan pl, int seq_major, int score_fn, float* __restrict__ colsum,
             int32_t* __restrict__ cnt, int* status) {
  __shared__ float wsum[8][kMaxE];
  __shared__ int hist[kMaxE];
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  for (int e = threadIdx.x; e < E; e += blockDim.x) hist[e] = 0;
  __syncthreads();
  const int64_t blk = blockIdx.x;
  const int64_t b = blk / pl.cps, cidx = blk - b * pl.cps;
  const int64_t s0 = cidx * pl.chunk;
  int64_t s1 = s0 + pl.chunk;
  if (s1 > pl.S) s1 = pl.S;
  float col[EPL];
#pragma unroll
  for (int i = 0; i < EPL; ++i) col[i] = 0.f;
  for (int64_t s = s0 + warp; s < s1; s += 8) {
    const int64_t t = seq_token(b, s, pl.B, pl.S, seq_major);
    if (colsum != nullptr) {
      float p[EPL], sc[EPL], l[EPL];
      token_probs<EPL>(logits + t * E, E, score_fn, lane, p, sc, l);
#pragma unroll
      for (int i = 0; i < EPL; ++i) col[i] += p[i];
    }
    if (lane < k) {
      const int e = idx[t * k + lane];
      if (e >= 0 && e < E) atomicAdd(&hist[e], 1);
      else record_error(status, MOE_ERR_DEVICE_INDEX, (int)t);
    }
  }
  if (colsum != nullptr) {
#pragma unroll
    for (int i = 0; i < EPL; ++i) {
      const int e = lane + 32 * i;
      if (e < E) wsum[warp][e] = col[i];
    }
  }
  __syncthreads();
  for (int e = threadIdx.x; e < E; e += blockDim.x) {
    if (colsum != nullptr) {
      float v = 0.f;
#pragma unroll
      for (int w = 0; w < 8; ++w) v += wsum[w][e];
      colsum[blk * E + e] = v;
    }
    cnt[blk * E + e] = hist[e];
  }
}

// one CTA per sequence: its loss (fp64), and its counts summed over chunks
__global__ void __launch_bounds__(256)
seq_per_sequence(const float* __restrict__ colsum, const int32_t* __restrict__ cnt, int E, int k,
                 SeqPlan pl, float coeff, double* __restrict__ loss_b,
                 int32_t* __restrict__ cnt_b) {
  __shared__ double term[kMaxE];
  const int64_t b = blockIdx.x;
  for (int e = threadIdx.x; e < E; e += blockDim.x) {
    double cs = 0.0;
    int64_t n = 0;
    for (int64_t c = 0; c < pl.cps; ++c) {
      const int64_t r = (b * pl.cps + c) * E + e;
      if (colsum != nullptr) cs += (double)colsum[r];
      n += cnt[r];
    }
    term[e] = cs * (double)n;
    if (cnt_b != nullptr) cnt_b[b * E + e] = (int32_t)n;
  }
  __syncthreads();
  if (threadIdx.x == 0 && loss_b != nullptr) {
    double acc = 0.0;
    for (int e = 0; e < E; ++e) acc += term[e];
    const double S = (double)pl.S;
    loss_b[b] = acc * (double)coeff * (double)E / ((double)k * S * S);
  }
}

__global__ void seq_mean(const double* __restrict__ loss_b, int64_t B, float* __restrict__ out) {
  if (threadIdx.x != 0 || blockIdx.x != 0) return;
  double v = 0.0;
  for (int64_t b = 0; b < B; ++b) v += loss_b[b];
  *out = (B > 0) ? (float)(v / (double)B) : 0.f;
}

template <int EPL>
__global__ void __launch_bounds__(256)
seq_bwd_kernel(const float* __restrict__ logits, const int32_t* __restrict__ cnt_b, int E,
               int score_fn, SeqPlan pl, int seq_major, float g_scale,
               float* __restrict__ d_logits, int accumulate) {
  const int lane = threadIdx.x & 31;
  const int64_t T = pl.B * pl.S;
  const int64_t nwarps = ((int64_t)gridDim.x * blockDim.x) >> 5;
  for (int64_t t = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5; t < T; t += nwarps) {
    const int64_t b = seq_major ? t % pl.B : t / pl.S;
    float p[EPL], s[EPL], l[EPL], dP[EPL];
    const float S = token_probs<EPL>(logits + t * E, E, score_fn, lane, p, s, l);
#pragma unroll
    for (int i = 0; i < EPL; ++i) {
      const int e = lane + 32 * i;
      dP[i] = (e < E) ? g_scale * (float)cnt_b[b * E + e] : 0.f;
    }
    float dot = 0.f;
#pragma unroll
    for (int i = 0; i < EPL; ++i) dot += p[i] * dP[i];
    dot = warp_sum(dot);
#pragma unroll
    for (int i = 0; i < EPL; ++i) {
      const int e = lane + 32 * i;
      if (e < E) {
        float g;
        if (score_fn == MOE_SCORE_SOFTMAX || score_fn == MOE_SCORE_SOFTMAX_PRE)
          g = p[i] * (dP[i] - dot);
        else
          g = (dP[i] - dot) / S * bias_score_deriv(l[i], s[i], score_fn);
        float* dst = d_logits + t * E + e;
        *dst = accumulate ? *dst + g : g;
      }
    }
  }
}

struct SeqWs {
  float* colsum;
  int32_t* cnt;
  double* loss_b;
  int32_t* cnt_b;
};

static SeqWs seq_ws(const moe_cfg& cfg, const SeqPlan& p, void* ws) {
  const size_t n = (size_t)(p.B * p.cps) * (size_t)cfg.E;
  uint8_t* base = static_cast<uint8_t*>(ws);
  SeqWs w;
  w.colsum = reinterpret_cast<float*>(base);
  base += (n * sizeof(float) + 255) & ~(size_t)255;
  w.cnt = reinterpret_cast<int32_t*>(base);
  base += (n * sizeof(int32_t) + 255) & ~(size_t)255;
  w.loss_b = reinterpret_cast<double*>(base);
  base += ((size_t)p.B * sizeof(double) + 255) & ~(size_t)255;
  w.cnt_b = reinterpret_cast<int32_t*>(base);
  return w;
}

cudaError_t launch_seq_aux_loss(const Ctx& c, const moe_cfg& cfg, const float* logits,
                                const int32_t* idx, int64_t S, int seq_major, float coeff,
                                float* out, void* ws) {
  const SeqPlan pl = seq_plan(cfg, S);
  const SeqWs w = seq_ws(cfg, pl, ws);
  const int epl = (cfg.E + 31) / 32;
  const unsigned nblk = (unsigned)(pl.B * pl.cps);
#define MOE_SP(N)                                                                          \
  seq_partials<N><<<nblk, 256, 0, c.stream>>>(logits, idx, cfg.E, cfg.k, pl, seq_major,   \
                                              cfg.score_fn, w.colsum, w.cnt, c.status)
  MOE_BY_EPL(epl, MOE_SP)
#undef MOE_SP
  seq_per_sequence<<<(unsigned)pl.B, 256, 0, c.stream>>>(w.colsum, w.cnt, cfg.E, cfg.k, pl,
                                                          coeff, w.loss_b, nullptr);
  seq_mean<<<1, 32, 0, c.stream>>>(w.loss_b, pl.B, out);
  note_launches(3);
  return cudaGetLastError();
}

cudaError_t launch_seq_aux_loss_bwd(const Ctx& c, const moe_cfg& cfg, const float* logits,
                                    const int32_t* idx, int64_t S, int seq_major, float coeff,
                                    float g, float* d_logits, int accumulate, void* ws) {
  const SeqPlan pl = seq_plan(cfg, S);
  const SeqWs w = seq_ws(cfg, pl, ws);
  const int epl = (cfg.E + 31) / 32;
  const unsigned nblk = (unsigned)(pl.B * pl.cps);
#define MOE_SC(N)                                                                          \
  seq_partials<N><<<nblk, 256, 0, c.stream>>>(logits, idx, cfg.E, cfg.k, pl, seq_major,   \
                                              cfg.score_fn, nullptr, w.cnt, c.status)
  MOE_BY_EPL(epl, MOE_SC)
#undef MOE_SC
  seq_per_sequence<<<(unsigned)pl.B, 256, 0, c.stream>>>(nullptr, w.cnt, cfg.E, cfg.k, pl, coeff,
                                                          nullptr, w.cnt_b);
  const double Sd = (double)S;
  const float g_scale = (float)((double)g * (double)coeff * (double)cfg.E /
                                ((double)cfg.k * Sd * Sd * (double)pl.B));
  const int64_t blocks = (cfg.T + 7) / 8;
  const int64_t cap = (int64_t)c.sm_count * 8;
  const unsigned grid = (unsigned)(blocks < cap ? blocks : cap);
#define MOE_SB(N)                                                                        \
  seq_bwd_kernel<N><<<grid, 256, 0, c.stream>>>(logits, w.cnt_b, cfg.E, cfg.score_fn, pl, \
                                                seq_major, g_scale, d_logits, accumulate)
  MOE_BY_EPL(epl, MOE_SB)
#undef MOE_SB
  note_launches(3);
  return cudaGetLastError();
}

cudaError_t launch_aux_loss(const Ctx& c, const moe_cfg& cfg, const float* logits,
                            const int32_t* counts, float* aux, void* ws) {
  const int64_t nblk = aux_blocks(cfg.T);
  float* part = static_cast<float*>(ws);
  const int epl = (cfg.E + 31) / 32;
  if (nblk > 0 && cfg.E <= 16) {
    if (cfg.E <= 8)
      launch_dependent(aux_partials_grouped<8>, dim3((unsigned)nblk), dim3(256), 0, c.stream,
                       logits, cfg.T, cfg.E, cfg.score_fn, part);
    else
      launch_dependent(aux_partials_grouped<16>, dim3((unsigned)nblk), dim3(256), 0, c.stream,
                       logits, cfg.T, cfg.E, cfg.score_fn, part);
  } else if (nblk > 0) {
#define MOE_AUXP(N)                                                                  \
  launch_dependent(aux_partials<N>, dim3((unsigned)nblk), dim3(256), 0, c.stream, logits, \
                   cfg.T, cfg.E, cfg.score_fn, part)
    switch (epl) {
      case 1: MOE_AUXP(1); break;
      case 2: MOE_AUXP(2); break;
      case 3: case 4: MOE_AUXP(4); break;
      default: MOE_AUXP(8); break;
    }
#undef MOE_AUXP
  }
  launch_dependent(aux_finalize, dim3(1), dim3(1024), 0, c.stream, part, nblk, counts, cfg.T,
                   cfg.E, cfg.k, cfg.aux_coeff, aux);
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
#define MOE_AUXB(N)                                                                       \
  launch_dependent(aux_bwd_kernel<N>, dim3(grid), dim3(256), 0, c.stream, logits, counts,    \
                   cfg.T, cfg.E, cfg.k, cfg.score_fn, g_scale, d_logits, accumulate)
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
