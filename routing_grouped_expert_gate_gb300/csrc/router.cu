// Router: gate GEMM (S1), scores + sorted top-k + mixing weights (S2), and the
// score backward (B2).
//
// The Ultimate MoE Training Handbook, §3.1 "Router scoring": logits come from
// an fp32 GEMM of the token with the [E, d] fp32 router weight ("Precision");
// softmax routing picks the top-k logits and takes the softmax over them,
// sigmoid routing picks on sigmoid(l) + expert bias and divides the chosen
// scores by their sum + 1e-20 ("Gating function", "Output scale"), then the
// routed scaling factor multiplies the weights. §3.2 "Who selects": the top-k
// is sorted.
//
// Accuracy: each logit is a sum of d products. The kernels add the products of
// one 32-element chunk in plain fp32 FMAs and fold the chunk sums into a
// (hi, lo) pair with an error-free TwoSum, so the only rounding that grows with
// d is confined to 32-term partial sums. The logits end within a few fp32 ulps
// of the exact value, far inside the 1e-6 band that marks a near tie.
#include <type_traits>

#include "common.cuh"
#include "lane_groups.cuh"
#include "internal.h"
#include "tc_ptx.cuh"

namespace moe {

// ------------------------------------------------------------------ S1, E <= 16
// One CTA per TB tokens. The 8 warps split the hidden dimension into eight
// ranges of 8-element groups; lane l of warp w reads groups l, l+32, ... of
// range w, so a token row is read once, 16 B per lane at a time, and every W
// value a lane loads serves the CTA's TB tokens. Per lane, the products of up
// to four groups (32 elements) are added in fp32 FMAs and folded into a
// compensated (hi, lo) pair; the pairs are combined by a reduce-scatter over
// the lanes and then over the warps in warp order, every step a TwoSum, so the
// result does not depend on scheduling. FOLD = false when no lane has more than
// four groups (d <= 8192): its fp32 sum is then the chunk sum itself.
template <typename Tx, int EMAX, int TB, bool FOLD>
__global__ void __launch_bounds__(256)
router_logits_small(const Tx* __restrict__ x, const float* __restrict__ W,
                    const float* __restrict__ logit_bias, float* __restrict__ logits,
                    int64_t T, int d, int E) {
  __shared__ float s_hi[8][TB * EMAX];
  __shared__ float s_lo[8][TB * EMAX];
  const int lane = threadIdx.x & 31;
  const int warp = threadIdx.x >> 5;
  const int64_t t0 = (int64_t)blockIdx.x * TB;
  const int ngroups = d >> 3;
  const int g_lo = (int)((int64_t)ngroups * warp / 8);
  const int g_hi = (int)((int64_t)ngroups * (warp + 1) / 8);

  float hi[TB][EMAX], lo[TB][EMAX], acc[TB][EMAX];
#pragma unroll
  for (int a = 0; a < TB; ++a)
#pragma unroll
    for (int e = 0; e < EMAX; ++e) acc[a][e] = 0.f;
  if (FOLD) {
#pragma unroll
    for (int a = 0; a < TB; ++a)
#pragma unroll
      for (int e = 0; e < EMAX; ++e) hi[a][e] = lo[a][e] = 0.f;
  }

  int cnt = 0;
  for (int g = g_lo + lane; g < g_hi; g += 32) {
    float xv[TB][8];
#pragma unroll
    for (int a = 0; a < TB; ++a) {
      if (t0 + a < T) {
        load8(x + (t0 + a) * (int64_t)d + 8 * g, xv[a]);
      } else {
#pragma unroll
        for (int i = 0; i < 8; ++i) xv[a][i] = 0.f;
      }
    }
#pragma unroll
    for (int e = 0; e < EMAX; ++e) {
      if (e < E) {
        float wv[8];
        load8(W + (int64_t)e * d + 8 * g, wv);
#pragma unroll
        for (int a = 0; a < TB; ++a)
#pragma unroll
          for (int i = 0; i < 8; ++i) acc[a][e] = fmaf(xv[a][i], wv[i], acc[a][e]);
      }
    }
    if (FOLD && ++cnt == 4) {  // 32 elements per lane
#pragma unroll
      for (int a = 0; a < TB; ++a)
#pragma unroll
        for (int e = 0; e < EMAX; ++e) {
          comp_add(hi[a][e], lo[a][e], acc[a][e]);
          acc[a][e] = 0.f;
        }
      cnt = 0;
    }
  }
#pragma unroll
  for (int a = 0; a < TB; ++a)
#pragma unroll
    for (int e = 0; e < EMAX; ++e) {
      if (FOLD) {
        comp_add(hi[a][e], lo[a][e], acc[a][e]);
      } else {
        hi[a][e] = acc[a][e];
        lo[a][e] = 0.f;
      }
    }

  // Reduce-scatter over the lanes: at each halving step a lane keeps one half
  // of its pairs (the upper half when its lane bit is set), gives the other
  // half to its partner and adds what it receives with a TwoSum, so lane q
  // ends with the warp's sum of pair q = a * EMAX + e (31 exchanges per lane
  // instead of 5 x 32 for a full butterfly).
  static_assert(TB * EMAX == 32, "one pair per lane after the reduce-scatter");
  float vh[32], vl[32];
#pragma unroll
  for (int a = 0; a < TB; ++a)
#pragma unroll
    for (int e = 0; e < EMAX; ++e) {
      vh[a * EMAX + e] = hi[a][e];
      vl[a * EMAX + e] = lo[a][e];
    }
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) {
    const bool upper = (lane & off) != 0;
#pragma unroll
    for (int q = 0; q < off; ++q) {
      const float sh_ = upper ? vh[q] : vh[q + off];
      const float sl_ = upper ? vl[q] : vl[q + off];
      const float kh = upper ? vh[q + off] : vh[q];
      const float kl = upper ? vl[q + off] : vl[q];
      const float rh = __shfl_xor_sync(0xffffffffu, sh_, off);
      const float rl = __shfl_xor_sync(0xffffffffu, sl_, off);
      float s2, er;
      two_sum(kh, rh, s2, er);
      vh[q] = s2;
      vl[q] = __fadd_rn(__fadd_rn(kl, rl), er);
    }
  }
  s_hi[warp][lane] = vh[0];
  s_lo[warp][lane] = vl[0];
  __syncthreads();
  // the eight warp partials of one logit, in warp order
  for (int q = threadIdx.x; q < TB * EMAX; q += blockDim.x) {
    const int a = q / EMAX, e = q - a * EMAX;
    if (e >= E || t0 + a >= T) continue;
    float h = s_hi[0][q], l = s_lo[0][q];
#pragma unroll
    for (int w = 1; w < 8; ++w) {
      float s2, er;
      two_sum(h, s_hi[w][q], s2, er);
      h = s2;
      l = __fadd_rn(__fadd_rn(l, s_lo[w][q]), er);
    }
    if (logit_bias != nullptr) comp_add(h, l, logit_bias[e]);
    logits[(t0 + a) * (int64_t)E + e] = __fadd_rn(h, l);
  }
}

// The lanes of a warp each hold TB x EMAX compensated (hi, lo) pairs of the
// same TB tokens (TB * EMAX = 32 or 16), partial sums over different elements.
// A reduce-scatter over the lanes (at each halving step a lane keeps one half
// of its pairs, gives the other half to its partner and adds what it receives
// with a TwoSum) leaves lane q with pair q = (token q / EMAX, expert q % EMAX)
// (with 16 pairs, lanes 2q and 2q + 1 with pair q, which they then add the
// same way), which it rounds once (after the logit bias) and stores.
template <int TB, int EMAX>
__device__ __forceinline__ void store_pair_logits(const float (&hi)[TB][EMAX],
                                                  const float (&lo)[TB][EMAX], int64_t t0,
                                                  int64_t T, int E,
                                                  const float* __restrict__ logit_bias,
                                                  float* __restrict__ logits) {
  constexpr int N = TB * EMAX;
  static_assert(N == 32 || N == 16, "one pair per lane or lane pair after the reduce-scatter");
  const int lane = threadIdx.x & 31;
  float vh[N], vl[N];
#pragma unroll
  for (int a = 0; a < TB; ++a)
#pragma unroll
    for (int e = 0; e < EMAX; ++e) {
      vh[a * EMAX + e] = hi[a][e];
      vl[a * EMAX + e] = lo[a][e];
    }
#pragma unroll
  for (int off = N / 2, bit = 16; off > 0; off >>= 1, bit >>= 1) {
    const bool upper = (lane & bit) != 0;
#pragma unroll
    for (int q = 0; q < off; ++q) {
      const float sh_ = upper ? vh[q] : vh[q + off];
      const float sl_ = upper ? vl[q] : vl[q + off];
      const float kh = upper ? vh[q + off] : vh[q];
      const float kl = upper ? vl[q + off] : vl[q];
      const float rh = __shfl_xor_sync(0xffffffffu, sh_, bit);
      const float rl = __shfl_xor_sync(0xffffffffu, sl_, bit);
      float s2, er;
      two_sum(kh, rh, s2, er);
      vh[q] = s2;
      vl[q] = __fadd_rn(__fadd_rn(kl, rl), er);
    }
  }
  int q = lane;
  if constexpr (N == 16) {
    const float rh = __shfl_xor_sync(0xffffffffu, vh[0], 1);
    const float rl = __shfl_xor_sync(0xffffffffu, vl[0], 1);
    float s2, er;
    two_sum(vh[0], rh, s2, er);
    vh[0] = s2;
    vl[0] = __fadd_rn(__fadd_rn(vl[0], rl), er);
    q = lane >> 1;
  }
  const int a = q / EMAX, e = q - a * EMAX;
  if ((N == 32 || (lane & 1) == 0) && e < E && t0 + a < T) {
    float h = vh[0], l = vl[0];
    if (logit_bias != nullptr) comp_add(h, l, logit_bias[e]);
    logits[(t0 + a) * (int64_t)E + e] = __fadd_rn(h, l);
  }
}

// ------------------------------------------------------------------ S1, E <= 16, W resident
// W stays in shared memory for the kernel's life ([E][2][d/8] float4 planes,
// staged once per CTA) and every warp works alone on groups of TB tokens, one
// CTA per SM walking the token groups: no block-wide barrier per group, so the
// eight warps' loads and arithmetic overlap. A lane takes the 8-element groups
// lane, lane + 32, ... of the hidden dimension in chunks of CH = 2 groups: the
// next chunk's x loads are issued before the current chunk's products with W
// (read from shared memory, consecutive words across the lanes) are summed in
// plain fp32 FMAs (16 elements) and folded into a compensated (hi, lo) pair
// per (token, expert). The lanes' pairs are then combined by a reduce-scatter with
// TwoSums (lane q ends with pair q = token q / EMAX, expert q % EMAX), so each
// logit carries only the rounding of its 32-element chunk sums.
template <typename Tx, int EMAX, int TB>
__global__ void __launch_bounds__(256, 1)
router_logits_resident(const Tx* __restrict__ x, const float* __restrict__ W,
                       const float* __restrict__ logit_bias, float* __restrict__ logits,
                       int64_t T, int d, int E) {
  extern __shared__ float4 sW[];  // [E][2][ngroups]
  static_assert(TB * EMAX == 32, "one pair per lane after the reduce-scatter");
  constexpr int CH = 2;  // groups of 8 per chunk: 16 elements per plain-fp32 chunk sum
  pdl_wait();  // x may come from the kernel before; logits may still be read by it
  const int lane = threadIdx.x & 31;
  const int ngroups = d >> 3;
  const int64_t n_tg = (T + TB - 1) / TB;
  const int64_t warps = (int64_t)gridDim.x * (blockDim.x >> 5);

  // the warp walks (token group, chunk) positions; the next position's x is
  // loaded while the current one is multiplied
  // (gb is warp-uniform: the chunk's first group; lane takes gb + lane + 32 c)
  auto load_chunk = [&](int64_t tg, int gb, Raw8<Tx> (&buf)[CH][TB]) {
    const int64_t t0 = tg * TB;
#pragma unroll
    for (int c = 0; c < CH; ++c) {
      const int g = gb + lane + 32 * c;
#pragma unroll
      for (int a = 0; a < TB; ++a) {
        if (g < ngroups && t0 + a < T) buf[c][a].load(x + (t0 + a) * (int64_t)d + 8 * g);
        else buf[c][a].zero();
      }
    }
  };
  int64_t tg = (int64_t)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
  int gb = 0;
  Raw8<Tx> cur[CH][TB], nxt[CH][TB];
  if (tg < n_tg) load_chunk(tg, gb, cur);  // in flight while W is staged
  stage_w_planes(sW, W, E, d);

  float hi[TB][EMAX], lo[TB][EMAX];
  while (tg < n_tg) {
    int64_t tg_n = tg;
    int gb_n = gb + 32 * CH;
    if (gb_n >= ngroups) {
      tg_n = tg + warps;
      gb_n = 0;
    }
    if (tg_n < n_tg) load_chunk(tg_n, gb_n, nxt);
    if (gb == 0) {
#pragma unroll
      for (int a = 0; a < TB; ++a)
#pragma unroll
        for (int e = 0; e < EMAX; ++e) hi[a][e] = lo[a][e] = 0.f;
    }
    float acc[TB][EMAX];
#pragma unroll
    for (int a = 0; a < TB; ++a)
#pragma unroll
      for (int e = 0; e < EMAX; ++e) acc[a][e] = 0.f;
#pragma unroll
    for (int c = 0; c < CH; ++c) {
      const int g = gb + lane + 32 * c;
      if (g >= ngroups) continue;
      float xv[TB][8];
#pragma unroll
      for (int a = 0; a < TB; ++a) cur[c][a].to_float(xv[a]);
#pragma unroll
      for (int e = 0; e < EMAX; ++e) {
        if (e < E) {
          const float4 w0 = sW[(e * 2) * ngroups + g];
          const float4 w1 = sW[(e * 2 + 1) * ngroups + g];
          const float wv[8] = {w0.x, w0.y, w0.z, w0.w, w1.x, w1.y, w1.z, w1.w};
#pragma unroll
          for (int a = 0; a < TB; ++a)
#pragma unroll
            for (int i = 0; i < 8; ++i) acc[a][e] = fmaf(xv[a][i], wv[i], acc[a][e]);
        }
      }
    }
#pragma unroll
    for (int a = 0; a < TB; ++a)
#pragma unroll
      for (int e = 0; e < EMAX; ++e) comp_add(hi[a][e], lo[a][e], acc[a][e]);

    if (tg_n != tg) store_pair_logits<TB, EMAX>(hi, lo, tg * TB, T, E, logit_bias, logits);
#pragma unroll
    for (int c = 0; c < CH; ++c)
#pragma unroll
      for (int a = 0; a < TB; ++a) cur[c][a] = nxt[c][a];
    tg = tg_n;
    gb = gb_n;
  }
}

// Shared memory the resident form may take for W (E x d fp32).
constexpr size_t kRouterResidentSmem = 160 * 1024;

template <typename Tx, int EMAX, int TB>
static cudaError_t launch_router_resident(const Ctx& c, const Tx* x, const float* w_router,
                                          const float* logit_bias, float* logits, int64_t T,
                                          int d, int E) {
  auto kern = router_logits_resident<Tx, EMAX, TB>;
  static bool attr_done[64];
  int dev = 0;
  cudaGetDevice(&dev);
  if (!attr_done[dev & 63]) {
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)kRouterResidentSmem);
    if (e != cudaSuccess) return e;
    attr_done[dev & 63] = true;
  }
  const int64_t n_tg = (T + TB - 1) / TB;
  const int64_t need = (n_tg + 7) / 8;  // eight warps per CTA
  const int64_t grid = need < c.sm_count ? need : c.sm_count;
  const size_t smem = (size_t)E * d * sizeof(float);
  return launch_dependent(kern, dim3((unsigned)grid), dim3(256), smem, c.stream, x, w_router,
                          logit_bias, logits, T, d, E);
}

// ------------------------------------------------------------------ S1, E <= 16, bf16 x streamed
// W_r stays in shared memory ([E][d] fp32, one bulk copy) and the tokens'
// rows stream through a ring of slots, each TBLK = 16 TB tokens x 256 columns,
// one TMA tile load per slot from a producer thread (rows past T and columns
// past d arrive as zeros): the bytes in flight per SM are bounded by the ring
// (up to 128 KB), not by registers. Sixteen consumer warps take TB = 16 / EMAX
// tokens each of every slot (the kernel is bound by instruction issue: eight
// warps of twice the tokens measured 23.8 us for the route call at T = 4096,
// d = 4096, E = 8, sixteen 22.4 us); lane l takes columns 4l..4l+3 and 128+4l..128+4l+3 (W and x read from shared memory
// at consecutive addresses across the lanes). Per slot a lane forms, for each
// of its tokens and each expert, a chain of 8 fp32 FMAs; every two slots (16
// elements) the chain folds into the (token, expert) compensated pair, and
// store_pair_logits combines the lanes' pairs at the end of the block. Every
// mbarrier wait is bounded (MOE_ERR_TIMEOUT + abort flag).
struct StreamParams {
  int64_t T;
  int d, E, ns;  // ns: ring slots
  const float* logit_bias;
  float* logits;
  int* status;
  uint64_t timeout_ns;
};

constexpr int kStreamThreads = 288;  // 8 consumer warps + 1 producer warp (dW_r stream)
constexpr int kLsConsumers = 16;     // consumer warps of the logits stream
constexpr int kLsThreads = 32 * (kLsConsumers + 1);  // + 1 producer warp
constexpr int kStreamCols = 256;     // columns per slot
constexpr int kStreamMaxSlots = 8;

template <int EMAX>
struct StreamTile {
  static constexpr int TB = 16 / EMAX;                   // tokens per consumer warp
  static constexpr int TBLK = kLsConsumers * TB;         // tokens per slot
  static constexpr int kSlot = TBLK * kStreamCols * 2;   // bytes (bf16)
};

template <int EMAX>
__global__ void __launch_bounds__(kLsThreads, 1)
router_logits_stream(const __grid_constant__ CUtensorMap tmX, const float* __restrict__ W,
                     const StreamParams P) {
  using ST = StreamTile<EMAX>;
  constexpr int TB = ST::TB;
  extern __shared__ __align__(128) uint8_t sm_raw[];
  __shared__ __align__(8) uint64_t full[kStreamMaxSlots], empty[kStreamMaxSlots], wbar;
  __shared__ int abort_flag;
  const size_t w_bytes = ((size_t)P.E * P.d * sizeof(float) + 127) & ~(size_t)127;
  float* sW = reinterpret_cast<float*>(sm_raw);
  uint8_t* ring = sm_raw + w_bytes;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int d = P.d, E = P.E, ns = P.ns;
  const int nsl = (d + kStreamCols - 1) / kStreamCols;
  const int64_t nblk = (P.T + ST::TBLK - 1) / ST::TBLK;

  if (threadIdx.x == 0) {
    abort_flag = 0;
    for (int s = 0; s < ns; ++s) {
      tc::mbar_init(&full[s], 1);
      tc::mbar_init(&empty[s], kLsConsumers);  // one arrival per consumer warp
    }
    tc::mbar_init(&wbar, 1);
    tc::fence_barrier_init();
  }
  __syncthreads();
  pdl_wait();  // x may come from the kernel before; logits may still be read by it

  if (warp == kLsConsumers) {
    // ---------------- producer (one thread): W once, then the ring
    if (lane == 0) {
      tc::prefetch_tmap(&tmX);
      const uint32_t wb = (uint32_t)((size_t)E * d * sizeof(float));
      tc::mbar_expect_tx(&wbar, wb);
      tc::bulk_load_1d(sW, W, wb, &wbar);
    }
    int slot = 0;
    uint32_t ph = 0;
    bool ok = true;
    for (int64_t b = blockIdx.x; b < nblk && ok && lane == 0; b += gridDim.x) {
      const int t0 = (int)(b * ST::TBLK);
      for (int j = 0; j < nsl; ++j) {
        if (!tc::mbar_wait(&empty[slot], ph ^ 1, abort_flag, P, 41)) { ok = false; break; }
        tc::mbar_expect_tx(&full[slot], (uint32_t)ST::kSlot);
        tc::tma_load_2d(ring + (size_t)slot * ST::kSlot, &tmX, &full[slot], j * kStreamCols, t0);
        if (++slot == ns) { slot = 0; ph ^= 1; }
      }
    }
    if (!ok && lane == 0) {
      // let the copies already in flight land before the CTA exits
      const uint64_t t_start = global_timer_ns();
      while (global_timer_ns() - t_start < 2000000ull) { }
    }
  } else {
    // ---------------- consumers
    bool ok = tc::mbar_wait(&wbar, 0, abort_flag, P, 42);
    int slot = 0;
    uint32_t ph = 0;
    for (int64_t b = blockIdx.x; b < nblk && ok; b += gridDim.x) {
      float hi[TB][EMAX], lo[TB][EMAX], acc[TB][EMAX];
#pragma unroll
      for (int a = 0; a < TB; ++a)
#pragma unroll
        for (int e = 0; e < EMAX; ++e) hi[a][e] = lo[a][e] = acc[a][e] = 0.f;
      for (int j = 0; j < nsl; ++j) {
        if (!tc::mbar_wait(&full[slot], ph, abort_flag, P, 43)) { ok = false; break; }
        const uint8_t* sl = ring + (size_t)slot * ST::kSlot + (size_t)warp * TB * (kStreamCols * 2);
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          const int cl = h * 128 + 4 * lane;  // column within the slot
          const int c = j * kStreamCols + cl;
          if (c < d) {
            float xv[TB][4];
#pragma unroll
            for (int a = 0; a < TB; ++a) {
              const uint2 r = *reinterpret_cast<const uint2*>(sl + a * (kStreamCols * 2) + cl * 2);
              const float2 f0 = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&r.x));
              const float2 f1 = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&r.y));
              xv[a][0] = f0.x; xv[a][1] = f0.y; xv[a][2] = f1.x; xv[a][3] = f1.y;
            }
#pragma unroll
            for (int e = 0; e < EMAX; ++e) {
              if (e < E) {
                const float4 wv = *reinterpret_cast<const float4*>(sW + (size_t)e * d + c);
#pragma unroll
                for (int a = 0; a < TB; ++a) {
                  acc[a][e] = fmaf(xv[a][0], wv.x, acc[a][e]);
                  acc[a][e] = fmaf(xv[a][1], wv.y, acc[a][e]);
                  acc[a][e] = fmaf(xv[a][2], wv.z, acc[a][e]);
                  acc[a][e] = fmaf(xv[a][3], wv.w, acc[a][e]);
                }
              }
            }
          }
        }
        __syncwarp();
        if (lane == 0) tc::mbar_arrive(&empty[slot]);
        if (++slot == ns) { slot = 0; ph ^= 1; }
        if ((j & 1) || j == nsl - 1) {
#pragma unroll
          for (int a = 0; a < TB; ++a)
#pragma unroll
            for (int e = 0; e < EMAX; ++e) {
              comp_add(hi[a][e], lo[a][e], acc[a][e]);
              acc[a][e] = 0.f;
            }
        }
      }
      if (!ok) break;
      store_pair_logits<TB, EMAX>(hi, lo, b * ST::TBLK + warp * TB, P.T, E, P.logit_bias,
                                  P.logits);
    }
  }
}

// Dynamic shared memory the streamed form may take (W and the ring; the
// barriers sit in static shared memory, within the 227 KB a CTA may hold).
constexpr size_t kStreamSmemMax = 226 * 1024;

// Ring slots for the streamed form (0: it does not apply).
template <int EMAX>
static int stream_slots(const moe_cfg& cfg) {
  const size_t w_bytes = ((size_t)cfg.E * cfg.d * sizeof(float) + 127) & ~(size_t)127;
  if (w_bytes + 2 * (size_t)StreamTile<EMAX>::kSlot > kStreamSmemMax) return 0;
  const size_t n = (kStreamSmemMax - w_bytes) / StreamTile<EMAX>::kSlot;
  return (int)(n < (size_t)kStreamMaxSlots ? n : (size_t)kStreamMaxSlots);
}

template <int EMAX>
static cudaError_t launch_router_stream(const Ctx& c, const moe_cfg& cfg, const bf16* x,
                                        const float* w_router, const float* logit_bias,
                                        float* logits, int ns) {
  auto kern = router_logits_stream<EMAX>;
  static bool attr_done[64];
  int dev = 0;
  cudaGetDevice(&dev);
  if (!attr_done[dev & 63]) {
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)kStreamSmemMax);
    if (e != cudaSuccess) return e;
    attr_done[dev & 63] = true;
  }
  StreamParams P{};
  P.T = cfg.T;
  P.d = cfg.d;
  P.E = cfg.E;
  P.ns = ns;
  P.logit_bias = logit_bias;
  P.logits = logits;
  P.status = c.status;
  P.timeout_ns = c.timeout_ns;
  const size_t w_bytes = ((size_t)cfg.E * cfg.d * sizeof(float) + 127) & ~(size_t)127;
  const size_t smem = w_bytes + (size_t)ns * StreamTile<EMAX>::kSlot;
  const int64_t nblk = (cfg.T + StreamTile<EMAX>::TBLK - 1) / StreamTile<EMAX>::TBLK;
  const int64_t grid = nblk < c.sm_count ? nblk : c.sm_count;
  CUtensorMap mx;
  if (!tc::make_map_bf16_plain(&mx, x, cfg.T, cfg.d, StreamTile<EMAX>::TBLK, kStreamCols))
    return cudaErrorInvalidValue;
  return launch_dependent(kern, dim3((unsigned)grid), dim3(kLsThreads), smem, c.stream, mx,
                          w_router, P);
}

// ------------------------------------------------------------------ S1, E > 16
// Register-tiled fp32 SIMT GEMM on 256-thread CTAs. A CTA computes BT tokens x
// 64 experts; its threads form KS = 128 / BT groups of 2*BT threads that split
// K: group g takes the 64-wide K chunks g, g + KS, g + 2 KS, ... A thread
// computes 4 tokens x 8 experts ({4tx..4tx+3} and {32+4tx..32+4tx+3}, so that
// the eight threads of one shared-memory phase read 128 consecutive bytes).
// Partial sums fold into the compensated (hi, lo) pair every 32 elements; at
// the end group 0 adds the other groups' pairs in group order (deterministic).
// Smaller BT (more K groups) gives more CTAs when T x E is small; with large
// T x E the 128-token tile is fastest (W staged once per 128 tokens).
constexpr int RT_BE = 64, RT_KC = 64, RT_THREADS = 256;

template <int BT>
struct RouterTile {
  static constexpr int kGroups = 128 / BT;
  static constexpr int kGroupThreads = 2 * BT;
  static constexpr int kXs = RT_KC * (BT + 4);
  static constexpr int kWs = RT_KC * (RT_BE + 4);
  static constexpr int kGroupFloats = kXs + kWs;
  static constexpr size_t kSmem = (size_t)kGroups * kGroupFloats * sizeof(float);
  static_assert((kGroups - 1) * kGroupThreads * 64 <= kGroups * kGroupFloats,
                "the partial (hi, lo) pairs must fit in the staging buffers");
};

template <typename Tx, int BT>
__global__ void __launch_bounds__(RT_THREADS, 2)
router_logits_tiled(const Tx* __restrict__ x, const float* __restrict__ W,
                    const float* __restrict__ logit_bias, float* __restrict__ logits,
                    int64_t T, int d, int E) {
  using RT = RouterTile<BT>;
  constexpr int KS = RT::kGroups;
  constexpr int NT = RT::kGroupThreads;
  extern __shared__ __align__(16) float rt_smem[];
  const int grp = threadIdx.x / NT;
  const int tid = threadIdx.x % NT;
  float* gbuf = rt_smem + grp * RT::kGroupFloats;
  float (*xs)[BT + 4] = reinterpret_cast<float (*)[BT + 4]>(gbuf);
  float (*ws)[RT_BE + 4] = reinterpret_cast<float (*)[RT_BE + 4]>(gbuf + RT::kXs);

  const int ty = tid >> 3;  // token group: tokens 4ty..4ty+3
  const int tx = tid & 7;   // expert group
  const int64_t t_base = (int64_t)blockIdx.x * BT;
  const int e_base = blockIdx.y * RT_BE;

  float acc[4][8], hi[4][8], lo[4][8];
#pragma unroll
  for (int i = 0; i < 4; ++i)
#pragma unroll
    for (int j = 0; j < 8; ++j) acc[i][j] = hi[i][j] = lo[i][j] = 0.f;

  // loader roles: x: 4 x (token v % BT, group kg = v / BT); W: 512 / NT x (expert v & 63, kg v >> 6)
  auto stage_chunk = [&](int k0) {
#pragma unroll
    for (int r = 0; r < (8 * BT) / NT; ++r) {
      const int v = tid + NT * r;
      const int tok = v % BT, kg = v / BT;
      const int64_t t = t_base + tok;
      const int kk = k0 + 8 * kg;
      float xr[8];
      if (t < T && kk < d) {
        load8(x + t * d + kk, xr);
      } else {
#pragma unroll
        for (int i = 0; i < 8; ++i) xr[i] = 0.f;
      }
#pragma unroll
      for (int i = 0; i < 8; ++i) xs[kg * 8 + i][tok] = xr[i];
    }
#pragma unroll
    for (int r = 0; r < 512 / NT; ++r) {
      const int v = tid + NT * r;
      const int e = v & 63, kg = v >> 6;
      const int kk = k0 + 8 * kg;
      float wr[8];
      if (e_base + e < E && kk < d) {
        load8(W + (int64_t)(e_base + e) * d + kk, wr);
      } else {
#pragma unroll
        for (int i = 0; i < 8; ++i) wr[i] = 0.f;
      }
#pragma unroll
      for (int i = 0; i < 8; ++i) ws[kg * 8 + i][e] = wr[i];
    }
  };

  const int n_chunks = (d + RT_KC - 1) / RT_KC;
  const int rounds = (n_chunks + KS - 1) / KS;
  for (int rd = 0; rd < rounds; ++rd) {
    const int chunk = rd * KS + grp;
    const bool mine = chunk < n_chunks;  // uniform within a group
    __syncthreads();
    if (mine) stage_chunk(chunk * RT_KC);
    __syncthreads();
    if (!mine) continue;
    // plain FMAs over 32 elements, then the partial sums fold into (hi, lo):
    // the rounding that grows with d stays inside 32-term partial sums
#pragma unroll
    for (int half = 0; half < RT_KC / 32; ++half) {
#pragma unroll
      for (int k2 = 0; k2 < 32; ++k2) {
        const int kk = half * 32 + k2;
        const float4 a = *reinterpret_cast<const float4*>(&xs[kk][4 * ty]);
        const float4 b0 = *reinterpret_cast<const float4*>(&ws[kk][4 * tx]);
        const float4 b1 = *reinterpret_cast<const float4*>(&ws[kk][32 + 4 * tx]);
        const float av[4] = {a.x, a.y, a.z, a.w};
        const float bv[8] = {b0.x, b0.y, b0.z, b0.w, b1.x, b1.y, b1.z, b1.w};
#pragma unroll
        for (int i = 0; i < 4; ++i)
#pragma unroll
          for (int j = 0; j < 8; ++j) acc[i][j] = fmaf(av[i], bv[j], acc[i][j]);
      }
#pragma unroll
      for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int j = 0; j < 8; ++j) {
          comp_add(hi[i][j], lo[i][j], acc[i][j]);
          acc[i][j] = 0.f;
        }
    }
  }

  if constexpr (KS > 1) {
    // groups 1..KS-1 park their pairs in the staging buffers; group 0 adds
    // them in group order
    __syncthreads();
    float* park = rt_smem;  // [KS-1][NT][64], thread-major within a group
    if (grp > 0) {
      float* mine = park + ((size_t)(grp - 1) * NT + tid) * 64;
#pragma unroll
      for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int j = 0; j < 8; ++j) {
          mine[(i * 8 + j) * 2] = hi[i][j];
          mine[(i * 8 + j) * 2 + 1] = lo[i][j];
        }
    }
    __syncthreads();
    if (grp > 0) return;
#pragma unroll 1
    for (int g = 1; g < KS; ++g) {
      const float* theirs = park + ((size_t)(g - 1) * NT + tid) * 64;
#pragma unroll
      for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int j = 0; j < 8; ++j) {
          comp_add(hi[i][j], lo[i][j], theirs[(i * 8 + j) * 2]);
          lo[i][j] += theirs[(i * 8 + j) * 2 + 1];
        }
    }
  }

#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const int64_t t = t_base + 4 * ty + i;
    if (t >= T) continue;
#pragma unroll
    for (int half = 0; half < 2; ++half) {
      const int e0 = e_base + 32 * half + 4 * tx;
      float v[4];
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        float h = hi[i][4 * half + j], l = lo[i][4 * half + j];
        if (logit_bias != nullptr && e0 + j < E) comp_add(h, l, logit_bias[e0 + j]);
        v[j] = __fadd_rn(h, l);
      }
      if (e0 + 3 < E && (E & 3) == 0) {
        *reinterpret_cast<float4*>(logits + t * E + e0) = make_float4(v[0], v[1], v[2], v[3]);
      } else {
#pragma unroll
        for (int j = 0; j < 4; ++j)
          if (e0 + j < E) logits[t * E + e0 + j] = v[j];
      }
    }
  }
}

template <typename Tx, int BT>
static cudaError_t launch_router_tiled(const Ctx& c, const Tx* x, const float* w_router,
                                       const float* logit_bias, float* logits, int64_t T, int d,
                                       int E) {
  constexpr size_t smem = RouterTile<BT>::kSmem;
  static bool attr_done[64];
  int dev = 0;
  cudaGetDevice(&dev);
  if (!attr_done[dev & 63]) {
    cudaError_t e = cudaFuncSetAttribute(router_logits_tiled<Tx, BT>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    attr_done[dev & 63] = true;
  }
  dim3 grid((unsigned)((T + BT - 1) / BT), (unsigned)((E + RT_BE - 1) / RT_BE));
  router_logits_tiled<Tx, BT><<<grid, RT_THREADS, smem, c.stream>>>(x, w_router, logit_bias,
                                                                     logits, T, d, E);
  return cudaSuccess;
}

// ------------------------------------------------------------------ S2 keys
// The values a token's top-k ranks, lane l holding experts l, l+32, ...:
// the logit (softmax), the probability under the softmax over all E
// (pre-softmax), or the score (sigmoid, sqrt(softplus)); then + the selection
// bias, or - the quantile bias; a NaN key ranks last (-inf); slots past E
// hold -inf. pre_max / pre_inv: the pre-softmax's maximum and 1 / sum. With
// G < 32 a token takes a group of G lanes (EPL = 1, E <= G), `lane` its lane
// in the group.
template <int EPL, int G = 32>
__device__ __forceinline__ void selection_keys(const float* __restrict__ lrow,
                                               const float* __restrict__ sel_bias,
                                               const float* __restrict__ beta, int E,
                                               int score_fn, int lane, float (&key)[EPL],
                                               float& pre_max, float& pre_inv) {
  float lg[EPL];
#pragma unroll
  for (int i = 0; i < EPL; ++i) {
    const int e = lane + 32 * i;
    if (e < E) {
      const float l = lrow[e];
      // pre-softmax: replaced by the probability below
      key[i] = (score_fn == MOE_SCORE_SOFTMAX || score_fn == MOE_SCORE_SOFTMAX_PRE)
                   ? l : bias_score(l, score_fn);
      lg[i] = l;
    } else {
      key[i] = -INFINITY;
      lg[i] = 0.f;
    }
  }
  pre_inv = 0.f;
  pre_max = 0.f;
  if (score_fn == MOE_SCORE_SOFTMAX_PRE) {
    float m = -INFINITY;
#pragma unroll
    for (int i = 0; i < EPL; ++i)
      if (lane + 32 * i < E) m = fmaxf(m, lg[i]);
    m = group_max<G>(m);
    float sum = 0.f;
#pragma unroll
    for (int i = 0; i < EPL; ++i)
      if (lane + 32 * i < E) sum += expf(lg[i] - m);
    sum = group_sum<G>(sum);
    pre_max = m;
    pre_inv = 1.f / sum;
#pragma unroll
    for (int i = 0; i < EPL; ++i)
      if (lane + 32 * i < E) key[i] = expf(lg[i] - m) * pre_inv;
  }
#pragma unroll
  for (int i = 0; i < EPL; ++i) {
    const int e = lane + 32 * i;
    if (e < E) {
      float kv = key[i];
      if (sel_bias != nullptr) kv = __fadd_rn(kv, sel_bias[e]);
      if (beta != nullptr) kv = __fsub_rn(kv, beta[e]);
      key[i] = (kv == kv) ? kv : -INFINITY;
    }
  }
}

// Sorts n = 1, 2, 4 or 8 values descending in registers with a fixed
// compare-exchange network (the 19-comparator network for 8 inputs; checked on
// every 0/1 input).
__device__ __forceinline__ void cas_desc(uint64_t& a, uint64_t& b) {
  const uint64_t hi = a > b ? a : b, lo = a > b ? b : a;
  a = hi;
  b = lo;
}
template <int N>
__device__ __forceinline__ void sort_desc(uint64_t (&v)[N]) {
  static_assert(N == 1 || N == 2 || N == 4 || N == 8, "network sizes");
  if constexpr (N == 2) {
    cas_desc(v[0], v[1]);
  } else if constexpr (N == 4) {
    cas_desc(v[0], v[1]); cas_desc(v[2], v[3]);
    cas_desc(v[0], v[2]); cas_desc(v[1], v[3]);
    cas_desc(v[1], v[2]);
  } else if constexpr (N == 8) {
    cas_desc(v[0], v[2]); cas_desc(v[1], v[3]); cas_desc(v[4], v[6]); cas_desc(v[5], v[7]);
    cas_desc(v[0], v[4]); cas_desc(v[1], v[5]); cas_desc(v[2], v[6]); cas_desc(v[3], v[7]);
    cas_desc(v[0], v[1]); cas_desc(v[2], v[3]); cas_desc(v[4], v[5]); cas_desc(v[6], v[7]);
    cas_desc(v[2], v[4]); cas_desc(v[3], v[5]);
    cas_desc(v[1], v[4]); cas_desc(v[3], v[6]);
    cas_desc(v[1], v[2]); cas_desc(v[3], v[4]); cas_desc(v[5], v[6]);
  }
}

// ------------------------------------------------------------------ S2
// One warp per token. Lane l holds experts l, l+32, ... The k winners are found
// by k rounds of a warp arg-max over (key descending, index ascending); a
// non-finite key counts as -inf so a valid expert always wins. With E <= G < 32
// a warp takes 32 / G tokens at once, a group of G lanes each, one expert per
// lane, and every reduction runs over the group (the same keys and order).
//
// Quantile routing (beta != NULL): the key is the score minus beta, k + 1
// experts are ranked, the first k are chosen and the (k+1)-th key is written
// to alpha[t] (the token's threshold).
template <int EPL, int G = 32>
__global__ void __launch_bounds__(256)
router_topk(const float* __restrict__ logits, const float* __restrict__ sel_bias,
            const float* __restrict__ beta, float* __restrict__ alpha,
            int32_t* __restrict__ idx, float* __restrict__ w, int64_t T, int E, int k,
            int score_fn, float scaling) {
  pdl_wait();  // the logits come from the kernel before
  static_assert(G == 32 || EPL == 1, "groups of G < 32 lanes hold one expert each");
  constexpr int SLOTS = 32 / G;  // tokens per warp at a time
  const int ksel = (alpha != nullptr) ? k + 1 : k;
  const int lane = threadIdx.x & (G - 1);  // the lane within the token's group
  const int slot = (threadIdx.x & 31) / G;
  const int64_t nwarps = ((int64_t)gridDim.x * blockDim.x) >> 5;
  for (int64_t tb = (((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5) * SLOTS; tb < T;
       tb += nwarps * SLOTS) {
    const int64_t t = tb + slot;
    const bool live = t < T;  // (a group past T still takes part in the shuffles)
    float key[EPL], pre_max, pre_inv;
    selection_keys<EPL, G>(logits + (live ? t : tb) * E, sel_bias, beta, E, score_fn, lane, key,
                           pre_max, pre_inv);
    // Each candidate as one 64-bit integer that orders like (key descending,
    // expert ascending): the key's bits made order-preserving as unsigned
    // (-0 counted as +0) above the complemented expert index; slots past E hold
    // 0, below every expert. Round j takes the warp's largest remaining value
    // (a butterfly max over the lanes' heads), its owner drops it, and lane j
    // keeps the winner's expert and key.
    uint64_t pk[EPL];
#pragma unroll
    for (int i = 0; i < EPL; ++i) {
      const int e = lane + 32 * i;
      if (e < E) {
        uint32_t b = __float_as_uint(key[i] + 0.f);
        b = (b & 0x80000000u) ? ~b : (b | 0x80000000u);
        pk[i] = ((uint64_t)b << 32) | (uint64_t)(~(uint32_t)e);
      } else {
        pk[i] = 0ull;
      }
    }
    // the lane's candidates sorted descending once, so that a round needs
    // only each lane's head: the winner's lane moves its next one up
    sort_desc<EPL>(pk);
    int my_e = 0;
    float my_key = 0.f;
#pragma unroll
    for (int j = 0; j < kMaxK + 1; ++j) {
      if (j < ksel) {
        uint64_t best = pk[0];
#pragma unroll
        for (int off = G / 2; off > 0; off >>= 1) {
          const uint64_t o = __shfl_xor_sync(0xffffffffu, best, off, G);
          best = o > best ? o : best;
        }
        if (pk[0] == best) {  // the one lane whose head won (values are distinct)
#pragma unroll
          for (int i = 0; i + 1 < EPL; ++i) pk[i] = pk[i + 1];
          pk[EPL - 1] = 0ull;
        }
        if (lane == j) {
          my_e = (int)(~(uint32_t)best);
          uint32_t b = (uint32_t)(best >> 32);
          b = (b & 0x80000000u) ? (b & 0x7fffffffu) : ~b;
          my_key = best == 0ull ? -INFINITY : __uint_as_float(b);
        }
      }
    }
    if (alpha != nullptr) {
      const float ak = __shfl_sync(0xffffffffu, my_key, k, G);
      if (lane == 0 && live) alpha[t] = ak;
    }
    // mixing weights: lane j < k weighs the j-th chosen expert
    const bool mine = lane < k && live;
    const float l_j = mine ? logits[t * E + my_e] : 0.f;
    float wj;
    if (score_fn == MOE_SCORE_SOFTMAX) {
      const float m = group_max<G>(mine ? l_j : -INFINITY);
      const float ex = mine ? expf(l_j - m) : 0.f;
      wj = ex * (scaling / group_sum<G>(ex));
    } else if (score_fn == MOE_SCORE_SOFTMAX_PRE) {
      wj = mine ? expf(l_j - pre_max) * pre_inv * scaling : 0.f;
    } else {
      const float sj = mine ? bias_score(l_j, score_fn) : 0.f;
      const float sum = group_sum<G>(sj);
      wj = sj * ((k > 1) ? scaling / (sum + 1e-20f) : scaling);
    }
    if (mine) {
      idx[t * k + lane] = my_e;
      w[t * k + lane] = wj;
    }
  }
}

// ------------------------------------------------------------------ S2 diagnostics
// Near ties: tokens whose k-th and (k+1)-th selection keys, the fp32 keys the
// top-k ranks (selection_keys), differ by less than `band`; for them the choice
// rests on rounding. One warp per token ranks k + 1 experts as router_topk
// does; each CTA adds its count to *count with one integer atomic, so the total
// does not depend on the order. Needs k < E.
template <int EPL>
__global__ void __launch_bounds__(256)
router_near_ties(const float* __restrict__ logits, const float* __restrict__ sel_bias, int64_t T,
                 int E, int k, int score_fn, float band, int* __restrict__ count) {
  __shared__ int s_cnt;
  if (threadIdx.x == 0) s_cnt = 0;
  __syncthreads();
  const int lane = threadIdx.x & 31;
  const int64_t nwarps = ((int64_t)gridDim.x * blockDim.x) >> 5;
  int mine = 0;
  for (int64_t t = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5; t < T; t += nwarps) {
    float key[EPL], pre_max, pre_inv;
    selection_keys<EPL>(logits + t * E, sel_bias, nullptr, E, score_fn, lane, key, pre_max,
                        pre_inv);
    uint64_t pk[EPL];
#pragma unroll
    for (int i = 0; i < EPL; ++i) {
      const int e = lane + 32 * i;
      if (e < E) {
        uint32_t b = __float_as_uint(key[i] + 0.f);
        b = (b & 0x80000000u) ? ~b : (b | 0x80000000u);
        pk[i] = ((uint64_t)b << 32) | (uint64_t)(~(uint32_t)e);
      } else {
        pk[i] = 0ull;
      }
    }
    float kth = 0.f, next = 0.f;
#pragma unroll
    for (int j = 0; j < kMaxK + 1; ++j) {
      if (j <= k) {
        uint64_t best = pk[0];
#pragma unroll
        for (int i = 1; i < EPL; ++i) best = pk[i] > best ? pk[i] : best;
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) {
          const uint64_t o = __shfl_xor_sync(0xffffffffu, best, off);
          best = o > best ? o : best;
        }
#pragma unroll
        for (int i = 0; i < EPL; ++i)
          if (pk[i] == best) pk[i] = 0ull;
        uint32_t b = (uint32_t)(best >> 32);
        b = (b & 0x80000000u) ? (b & 0x7fffffffu) : ~b;
        const float kv = best == 0ull ? -INFINITY : __uint_as_float(b);
        if (j == k - 1) kth = kv;
        if (j == k) next = kv;
      }
    }
    if (lane == 0 && __fsub_rn(kth, next) < band) ++mine;
  }
  if (lane == 0 && mine) atomicAdd(&s_cnt, mine);
  __syncthreads();
  if (threadIdx.x == 0 && s_cnt) atomicAdd(count, s_cnt);
}

// ------------------------------------------------------------------ B2
// d l_j for a token's k chosen logits lj[] from the upstream gradients gj[] of
// its mixing weights: the softmax over the chosen logits, or the normalised
// sigmoid-like scores (not the pre-softmax, where every logit moves).
__device__ __forceinline__ void chosen_logit_grads(const float (&lj)[kMaxK],
                                                   const float (&gj)[kMaxK], int k, int score_fn,
                                                   float scaling, float (&dl)[kMaxK]) {
  if (score_fn == MOE_SCORE_SOFTMAX) {
    float m = lj[0];
#pragma unroll
    for (int j = 1; j < kMaxK; ++j)
      if (j < k) m = fmaxf(m, lj[j]);
    float p[kMaxK], s = 0.f;
#pragma unroll
    for (int j = 0; j < kMaxK; ++j) {
      p[j] = (j < k) ? expf(lj[j] - m) : 0.f;
      s += p[j];
    }
    float dot = 0.f;
#pragma unroll
    for (int j = 0; j < kMaxK; ++j) {
      p[j] /= s;
      dot += p[j] * (scaling * gj[j]);
    }
#pragma unroll
    for (int j = 0; j < kMaxK; ++j) dl[j] = p[j] * (scaling * gj[j] - dot);
  } else {
    float sj[kMaxK], S = 0.f, dsd = 0.f;
#pragma unroll
    for (int j = 0; j < kMaxK; ++j) {
      sj[j] = (j < k) ? bias_score(lj[j], score_fn) : 0.f;
      S += sj[j];
      dsd += gj[j] * sj[j];
    }
    S += 1e-20f;
#pragma unroll
    for (int j = 0; j < kMaxK; ++j) {
      const float ds = (k > 1) ? scaling * (gj[j] - dsd / S) / S : scaling * gj[j];
      dl[j] = ds * bias_score_deriv(lj[j], sj[j], score_fn);
    }
  }
}

// One warp per token: zero the row (unless accumulating), then each of the
// first k lanes adds the gradient of its chosen logit.
__global__ void __launch_bounds__(256)
router_scores_bwd(const float* __restrict__ logits, const int32_t* __restrict__ idx,
                  const float* __restrict__ dw, float* __restrict__ d_logits, int64_t T,
                  int E, int k, int score_fn, float scaling, int accumulate, int* status) {
  pdl_wait();  // a dependent launch: inputs come from the kernels before
  const int lane = threadIdx.x & 31;
  const int64_t nwarps = ((int64_t)gridDim.x * blockDim.x) >> 5;
  for (int64_t t = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5; t < T; t += nwarps) {
    if (!accumulate)
      for (int e = lane; e < E; e += 32) d_logits[t * E + e] = 0.f;
    int ej[kMaxK];
    float lj[kMaxK], gj[kMaxK];
    bool ok = true;
#pragma unroll
    for (int j = 0; j < kMaxK; ++j) {
      ej[j] = 0;
      lj[j] = 0.f;
      gj[j] = 0.f;
      if (j < k) {
        int e = idx[t * k + j];
        if (e < 0 || e >= E) {
          ok = false;
          e = 0;
        }
        ej[j] = e;
        lj[j] = logits[t * E + e];
        gj[j] = dw[t * k + j];
      }
    }
    if (!ok) {
      if (lane == 0) record_error(status, MOE_ERR_DEVICE_INDEX, (int)t);
      continue;
    }
    float dl[kMaxK];
    if (score_fn == MOE_SCORE_SOFTMAX_PRE) {
      // w_j = c P[idx_j] with P the softmax over all E: every logit moves,
      // d l_e = c P_e (g_e - sum_j P[idx_j] dw_j)
      float m = -INFINITY;
      for (int e = lane; e < E; e += 32) m = fmaxf(m, logits[t * E + e]);
      m = warp_max(m);
      float sum = 0.f;
      for (int e = lane; e < E; e += 32) sum += expf(logits[t * E + e] - m);
      sum = warp_sum(sum);
      const float inv = 1.f / sum;
      float dot = 0.f;
#pragma unroll
      for (int j = 0; j < kMaxK; ++j)
        if (j < k) dot += expf(lj[j] - m) * inv * (scaling * gj[j]);
      for (int e = lane; e < E; e += 32) {
        float ge = 0.f;
#pragma unroll
        for (int j = 0; j < kMaxK; ++j)
          if (j < k && ej[j] == e) ge = scaling * gj[j];
        const float pe = expf(logits[t * E + e] - m) * inv;
        d_logits[t * E + e] += pe * (ge - dot);
      }
      continue;
    }
    chosen_logit_grads(lj, gj, k, score_fn, scaling, dl);
    __syncwarp();
#pragma unroll
    for (int j = 0; j < kMaxK; ++j)
      if (j < k && lane == j) d_logits[t * E + ej[j]] += dl[j];
  }
}


// The same for few experts and scores other than the pre-softmax: one thread
// per token (its k indices, logits and weight gradients loaded together), so
// that a warp takes 32 tokens instead of one.
__global__ void __launch_bounds__(256)
router_scores_bwd_rows(const float* __restrict__ logits, const int32_t* __restrict__ idx,
                       const float* __restrict__ dw, float* __restrict__ d_logits, int64_t T,
                       int E, int k, int score_fn, float scaling, int accumulate, int* status) {
  pdl_wait();  // a dependent launch: inputs come from the kernels before
  for (int64_t t = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; t < T;
       t += (int64_t)gridDim.x * blockDim.x) {
    int ej[kMaxK];
    float lj[kMaxK], gj[kMaxK], dl[kMaxK];
    bool ok = true;
#pragma unroll
    for (int j = 0; j < kMaxK; ++j) {
      ej[j] = 0;
      gj[j] = 0.f;
      if (j < k) {
        int e = idx[t * k + j];
        if (e < 0 || e >= E) {
          ok = false;
          e = 0;
        }
        ej[j] = e;
        gj[j] = dw[t * k + j];
      }
    }
#pragma unroll
    for (int j = 0; j < kMaxK; ++j) lj[j] = (j < k) ? logits[t * E + ej[j]] : 0.f;
    if (!ok) {
      record_error(status, MOE_ERR_DEVICE_INDEX, (int)t);
      continue;
    }
    chosen_logit_grads(lj, gj, k, score_fn, scaling, dl);
    float* row = d_logits + t * E;
    if (!accumulate)
      for (int e = 0; e < E; ++e) row[e] = 0.f;
#pragma unroll
    for (int j = 0; j < kMaxK; ++j)
      if (j < k) row[ej[j]] += dl[j];
  }
}

// ------------------------------------------------------------------ B3, E <= 16, bf16 x streamed
// dW_r partials for few experts, bf16 x: part[s][e][c] = sum over the tokens
// of slice s of d_logits[t][e] * x[t][c], from a TMA ring. A CTA takes 1024
// columns of one token slice (consumer thread i: columns 4i..4i+3). The
// slice's x rows stream through slots of 16 tokens x 1024 columns (four tile
// loads of 256 columns each, issued by a producer thread; columns past d
// arrive as zeros and are not used); the slice's d_logits rows sit in shared
// memory, padded to EMAX per token with zeros. A thread adds the tokens in
// order into EMAX x 4 fp32 sums; the slices are summed afterwards in slice
// order. Every mbarrier wait is bounded (MOE_ERR_TIMEOUT + abort flag).
constexpr int kDwCols = 1024, kDwTok = 16;
constexpr int kDwSlot = kDwTok * kDwCols * 2;  // 32 KB

struct DwParams {
  int64_t T;
  int d, E, ns;
  int tok_per_slice;
  float* part;
  int* status;
  uint64_t timeout_ns;
};

template <int EMAX>
__global__ void __launch_bounds__(kStreamThreads, 1)
router_dw_stream(const __grid_constant__ CUtensorMap tmX, const float* __restrict__ g,
                 const DwParams P) {
  static_assert(EMAX % 4 == 0, "d_logits rows read as float4");
  extern __shared__ __align__(128) uint8_t sm_raw[];
  __shared__ __align__(8) uint64_t full[kStreamMaxSlots], empty[kStreamMaxSlots];
  __shared__ int abort_flag;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int d = P.d, E = P.E, ns = P.ns;
  const int c0 = blockIdx.x * kDwCols;
  const int64_t t_beg = (int64_t)blockIdx.y * P.tok_per_slice;
  const int ntok = (int)(P.T - t_beg < P.tok_per_slice ? P.T - t_beg : P.tok_per_slice);
  const int nsl = (ntok + kDwTok - 1) / kDwTok;
  float* sg = reinterpret_cast<float*>(sm_raw);  // [tok_per_slice][EMAX]
  const size_t g_bytes = ((size_t)P.tok_per_slice * EMAX * sizeof(float) + 127) & ~(size_t)127;
  uint8_t* ring = sm_raw + g_bytes;

  if (threadIdx.x == 0) {
    abort_flag = 0;
    for (int s = 0; s < ns; ++s) {
      tc::mbar_init(&full[s], 1);
      tc::mbar_init(&empty[s], 8);  // one arrival per consumer warp
    }
    tc::fence_barrier_init();
  }
  __syncthreads();
  pdl_wait();  // a dependent launch: inputs come from the kernels before

  if (warp == 8) {
    // ---------------- producer (one thread)
    if (lane == 0) {
      tc::prefetch_tmap(&tmX);
      const int nbox = (d - c0 + 255) / 256 < 4 ? (d - c0 + 255) / 256 : 4;
      int slot = 0;
      uint32_t ph = 0;
      bool ok = true;
      for (int j = 0; j < nsl; ++j) {
        if (!tc::mbar_wait(&empty[slot], ph ^ 1, abort_flag, P, 44)) { ok = false; break; }
        tc::mbar_expect_tx(&full[slot], (uint32_t)(nbox * kDwSlot / 4));
        for (int k = 0; k < nbox; ++k)
          tc::tma_load_2d(ring + (size_t)slot * kDwSlot + k * (kDwSlot / 4), &tmX, &full[slot],
                          c0 + 256 * k, (int)(t_beg + j * kDwTok));
        if (++slot == ns) { slot = 0; ph ^= 1; }
      }
      if (!ok) {
        // let the copies already in flight land before the CTA exits
        const uint64_t t_start = global_timer_ns();
        while (global_timer_ns() - t_start < 2000000ull) { }
      }
    }
  } else {
    // ---------------- consumers (256 threads)
    const int tid = threadIdx.x;
    for (int i = tid; i < ntok * EMAX; i += 256) {
      const int t = i / EMAX, e = i - t * EMAX;
      sg[i] = e < E ? g[(t_beg + t) * E + e] : 0.f;
    }
    asm volatile("bar.sync 1, 256;" ::: "memory");  // the consumers only
    const int k = tid >> 6, cq = (tid & 63) * 4;
    const int col = c0 + 256 * k + cq;
    const bool active = col < d;
    float acc[EMAX][4];
#pragma unroll
    for (int e = 0; e < EMAX; ++e)
#pragma unroll
      for (int q = 0; q < 4; ++q) acc[e][q] = 0.f;
    bool ok = true;
    int slot = 0;
    uint32_t ph = 0;
    for (int j = 0; j < nsl; ++j) {
      if (!tc::mbar_wait(&full[slot], ph, abort_flag, P, 45)) { ok = false; break; }
      const int rows = ntok - j * kDwTok < kDwTok ? ntok - j * kDwTok : kDwTok;
      if (active) {
        const uint8_t* base = ring + (size_t)slot * kDwSlot + k * (kDwSlot / 4) + cq * 2;
        const float* gs = sg + (size_t)j * kDwTok * EMAX;
#pragma unroll 4
        for (int r = 0; r < rows; ++r) {
          const uint2 raw = *reinterpret_cast<const uint2*>(base + r * 512);
          const float2 f0 = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&raw.x));
          const float2 f1 = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&raw.y));
          const float xv[4] = {f0.x, f0.y, f1.x, f1.y};
#pragma unroll
          for (int e4 = 0; e4 < EMAX; e4 += 4) {
            const float4 gv = *reinterpret_cast<const float4*>(gs + r * EMAX + e4);
            const float gg[4] = {gv.x, gv.y, gv.z, gv.w};
#pragma unroll
            for (int u = 0; u < 4; ++u)
#pragma unroll
              for (int q = 0; q < 4; ++q) acc[e4 + u][q] = fmaf(gg[u], xv[q], acc[e4 + u][q]);
          }
        }
      }
      __syncwarp();
      if (lane == 0) tc::mbar_arrive(&empty[slot]);
      if (++slot == ns) { slot = 0; ph ^= 1; }
    }
    if (ok && active) {
      float* out = P.part + (int64_t)blockIdx.y * E * d;
#pragma unroll
      for (int e = 0; e < EMAX; ++e)
        if (e < E)
          *reinterpret_cast<float4*>(out + (int64_t)e * d + col) =
              make_float4(acc[e][0], acc[e][1], acc[e][2], acc[e][3]);
    }
  }
}

template <int EMAX>
static cudaError_t launch_router_dw_stream(const Ctx& c, const moe_cfg& cfg, const bf16* x,
                                           const float* d_logits, float* part, int tps,
                                           int n_ts) {
  auto kern = router_dw_stream<EMAX>;
  static bool attr_done[64];
  int dev = 0;
  cudaGetDevice(&dev);
  if (!attr_done[dev & 63]) {
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)kStreamSmemMax);
    if (e != cudaSuccess) return e;
    attr_done[dev & 63] = true;
  }
  const size_t g_bytes = ((size_t)tps * EMAX * sizeof(float) + 127) & ~(size_t)127;
  size_t ns = (kStreamSmemMax - g_bytes) / kDwSlot;
  if (ns > (size_t)kStreamMaxSlots) ns = kStreamMaxSlots;
  DwParams P{};
  P.T = cfg.T;
  P.d = cfg.d;
  P.E = cfg.E;
  P.ns = (int)ns;
  P.tok_per_slice = tps;
  P.part = part;
  P.status = c.status;
  P.timeout_ns = c.timeout_ns;
  CUtensorMap mx;
  if (!tc::make_map_bf16_plain(&mx, x, cfg.T, cfg.d, kDwTok, 256)) return cudaErrorInvalidValue;
  dim3 grid((unsigned)((cfg.d + kDwCols - 1) / kDwCols), (unsigned)n_ts);
  return launch_dependent(kern, grid, dim3(kStreamThreads), g_bytes + ns * kDwSlot, c.stream, mx,
                          d_logits, P);
}

// ------------------------------------------------------------------ B3, E <= 16
// dW_r partials for few experts: part[s][e][c] = sum over the tokens of slice s
// of d_logits[t][e] * x[t][c]. A thread owns 8 consecutive columns and every
// expert; the d_logits row of a token is the same for the whole CTA (a
// broadcast load). The tokens of a slice go in groups of U whose loads are
// issued together, and are added in token order. Slices are summed afterwards
// in slice order.
template <typename Tx, int EMAX>
__global__ void __launch_bounds__(128)
router_dw_small(const Tx* __restrict__ x, const float* __restrict__ d_logits,
                float* __restrict__ part, int64_t T, int d, int E, int64_t tok_per_slice) {
  pdl_wait();  // a dependent launch: inputs come from the kernels before
  constexpr int U = EMAX <= 8 ? 4 : 2;
  const int c0 = (blockIdx.x * 128 + threadIdx.x) * 8;
  const int64_t t_beg = (int64_t)blockIdx.y * tok_per_slice;
  const int64_t t_end = t_beg + tok_per_slice < T ? t_beg + tok_per_slice : T;
  if (c0 >= d) return;
  float acc[EMAX][8];
#pragma unroll
  for (int e = 0; e < EMAX; ++e)
#pragma unroll
    for (int i = 0; i < 8; ++i) acc[e][i] = 0.f;
  int64_t t = t_beg;
  for (; t + U <= t_end; t += U) {
    float xv[U][8], g[U][EMAX];
#pragma unroll
    for (int u = 0; u < U; ++u) {
      load8(x + (t + u) * d + c0, xv[u]);
#pragma unroll
      for (int e = 0; e < EMAX; ++e) g[u][e] = e < E ? __ldg(d_logits + (t + u) * E + e) : 0.f;
    }
#pragma unroll
    for (int u = 0; u < U; ++u)
#pragma unroll
      for (int e = 0; e < EMAX; ++e)
#pragma unroll
        for (int i = 0; i < 8; ++i) acc[e][i] = fmaf(g[u][e], xv[u][i], acc[e][i]);
  }
  for (; t < t_end; ++t) {
    float xv[8];
    load8(x + t * d + c0, xv);
#pragma unroll
    for (int e = 0; e < EMAX; ++e) {
      if (e < E) {
        const float g = __ldg(d_logits + t * E + e);
#pragma unroll
        for (int i = 0; i < 8; ++i) acc[e][i] = fmaf(g, xv[i], acc[e][i]);
      }
    }
  }
  float* out = part + (int64_t)blockIdx.y * E * d;
#pragma unroll
  for (int e = 0; e < EMAX; ++e)
    if (e < E) store8(out + (int64_t)e * d + c0, acc[e]);
}

cudaError_t launch_router_dw_small(const Ctx& c, const moe_cfg& cfg, const void* x,
                                   const float* d_logits, float* part, int splits, int* used) {
  *used = splits;
  if (cfg.T == 0) return cudaSuccess;
  if (cfg.act_dtype == MOE_BF16 && cfg.d % 8 == 0 && cfg.T <= (int64_t)INT32_MAX - 64 &&
      (reinterpret_cast<uintptr_t>(x) & 15) == 0) {
    // the streamed form: about one CTA per SM, token slices of a multiple of
    // 16 tokens whose padded d_logits rows take at most 32 KB
    const int emax = cfg.E <= 8 ? 8 : 16;
    const int64_t n_cs = (cfg.d + kDwCols - 1) / kDwCols;
    const int64_t want = c.sm_count / n_cs > 1 ? c.sm_count / n_cs : 1;
    int64_t tps = ((cfg.T + want - 1) / want + kDwTok - 1) / kDwTok * kDwTok;
    const int64_t cap = 8192 / emax;
    if (tps > cap) tps = cap;
    const int64_t n_ts = (cfg.T + tps - 1) / tps;
    if (n_ts <= splits) {
      cudaError_t e = emax == 8
          ? launch_router_dw_stream<8>(c, cfg, static_cast<const bf16*>(x), d_logits, part,
                                       (int)tps, (int)n_ts)
          : launch_router_dw_stream<16>(c, cfg, static_cast<const bf16*>(x), d_logits, part,
                                        (int)tps, (int)n_ts);
      if (e != cudaSuccess) return e;
      note_launches(1);
      *used = (int)n_ts;
      return cudaGetLastError();
    }
  }
  const int64_t per = (cfg.T + splits - 1) / splits;
  dim3 grid((unsigned)((cfg.d / 8 + 127) / 128), (unsigned)splits);
#define MOE_DWS(TX, EM)                                                                 \
  launch_dependent(router_dw_small<TX, EM>, dim3(grid), dim3(128), 0, c.stream,           \
                   static_cast<const TX*>(x), d_logits, part, cfg.T, cfg.d, cfg.E, per)
  if (cfg.act_dtype == MOE_BF16) {
    if (cfg.E <= 8) MOE_DWS(bf16, 8); else MOE_DWS(bf16, 16);
  } else {
    if (cfg.E <= 8) MOE_DWS(float, 8); else MOE_DWS(float, 16);
  }
#undef MOE_DWS
  note_launches(1);
  return cudaGetLastError();
}

// ------------------------------------------------------------------ B3 dx, E <= 16
// dx_router[t][c] = sum over e of d_logits[t][e] * W_r[e][c] (fp32, e in
// order). A thread keeps W_r's 4 consecutive columns for every expert in
// registers and walks the CTA's tokens; a warp writes 512 contiguous bytes of
// a row at a time. grid.x covers d in 1024-column chunks, grid.y the tokens in
// tiles of 32.
template <int EMAX>
__global__ void __launch_bounds__(256)
router_dx_small(const float* __restrict__ d_logits, const float* __restrict__ W,
                float* __restrict__ dx, int64_t T, int d, int E) {
  constexpr int TT = 32;
  const int c0 = (blockIdx.x * 256 + threadIdx.x) * 4;
  if (c0 >= d) return;
  float4 w[EMAX];
#pragma unroll
  for (int e = 0; e < EMAX; ++e)
    w[e] = e < E ? __ldg(reinterpret_cast<const float4*>(W + (int64_t)e * d + c0))
                 : make_float4(0.f, 0.f, 0.f, 0.f);
  const int64_t t_beg = (int64_t)blockIdx.y * TT;
  const int64_t t_end = t_beg + TT < T ? t_beg + TT : T;
  for (int64_t t = t_beg; t < t_end; ++t) {
    float4 o = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
    for (int e = 0; e < EMAX; ++e) {
      if (e < E) {
        const float g = __ldg(d_logits + t * E + e);
        o.x = fmaf(g, w[e].x, o.x);
        o.y = fmaf(g, w[e].y, o.y);
        o.z = fmaf(g, w[e].z, o.z);
        o.w = fmaf(g, w[e].w, o.w);
      }
    }
    *reinterpret_cast<float4*>(dx + t * d + c0) = o;
  }
}

cudaError_t launch_router_dx_small(const Ctx& c, const moe_cfg& cfg, const float* d_logits,
                                   const float* w_router, float* dx_router) {
  if (cfg.T == 0) return cudaSuccess;
  dim3 grid((unsigned)((cfg.d / 4 + 255) / 256), (unsigned)((cfg.T + 31) / 32));
  if (cfg.E <= 8)
    router_dx_small<8><<<grid, 256, 0, c.stream>>>(d_logits, w_router, dx_router, cfg.T, cfg.d,
                                                   cfg.E);
  else
    router_dx_small<16><<<grid, 256, 0, c.stream>>>(d_logits, w_router, dx_router, cfg.T,
                                                    cfg.d, cfg.E);
  note_launches(1);
  return cudaGetLastError();
}

// ------------------------------------------------------------------ launchers
template <typename Tx>
static cudaError_t router_logits_dispatch(const Ctx& c, const moe_cfg& cfg, const Tx* x,
                                          const float* w_router, const float* logit_bias,
                                          float* logits) {
  const int64_t T = cfg.T;
  if (T == 0) return cudaSuccess;
  if (cfg.E <= 16) {
    // groups of 8 per lane: d / 8 split over 8 warps of 32 lanes
    const bool fold = (cfg.d / 8 + 255) / 256 > 4;
    // bf16 x, W_r and a ring of at least two slots fit in shared memory, rows
    // and W_r 16-byte aligned: the streamed form
    if constexpr (std::is_same<Tx, bf16>::value) {
      const int ns = cfg.E <= 8 ? stream_slots<8>(cfg) : stream_slots<16>(cfg);
      if (ns >= 2 && cfg.d % 8 == 0 && cfg.T <= (int64_t)INT32_MAX - 64 &&
          (reinterpret_cast<uintptr_t>(x) & 15) == 0 &&
          (reinterpret_cast<uintptr_t>(w_router) & 15) == 0) {
        cudaError_t e = cfg.E <= 8
            ? launch_router_stream<8>(c, cfg, x, w_router, logit_bias, logits, ns)
            : launch_router_stream<16>(c, cfg, x, w_router, logit_bias, logits, ns);
        if (e != cudaSuccess) return e;
        note_launches(1);
        return cudaGetLastError();
      }
    }
    // W_r fits in shared memory: the resident form
    if ((size_t)cfg.E * cfg.d * sizeof(float) <= kRouterResidentSmem) {
      cudaError_t e = cfg.E <= 8
          ? launch_router_resident<Tx, 8, 4>(c, x, w_router, logit_bias, logits, T, cfg.d, cfg.E)
          : launch_router_resident<Tx, 16, 2>(c, x, w_router, logit_bias, logits, T, cfg.d,
                                              cfg.E);
      if (e != cudaSuccess) return e;
      note_launches(1);
      return cudaGetLastError();
    }
    const unsigned grid8 = (unsigned)((T + 3) / 4), grid16 = (unsigned)((T + 1) / 2);
    if (cfg.E <= 8 && !fold)
      router_logits_small<Tx, 8, 4, false><<<grid8, 256, 0, c.stream>>>(x, w_router, logit_bias,
                                                                        logits, T, cfg.d, cfg.E);
    else if (cfg.E <= 8)
      router_logits_small<Tx, 8, 4, true><<<grid8, 256, 0, c.stream>>>(x, w_router, logit_bias,
                                                                       logits, T, cfg.d, cfg.E);
    else if (!fold)
      router_logits_small<Tx, 16, 2, false><<<grid16, 256, 0, c.stream>>>(
          x, w_router, logit_bias, logits, T, cfg.d, cfg.E);
    else
      router_logits_small<Tx, 16, 2, true><<<grid16, 256, 0, c.stream>>>(
          x, w_router, logit_bias, logits, T, cfg.d, cfg.E);
  } else {
    // token tile: the largest that still gives every SM a CTA (a smaller tile
    // splits K inside the CTA and stages W once per fewer tokens)
    const int64_t e_tiles = (cfg.E + RT_BE - 1) / RT_BE;
    const int64_t sms = c.sm_count > 0 ? c.sm_count : 1;
    int best_bt = 32;
    for (int bt : {128, 64}) {
      if (((T + bt - 1) / bt) * e_tiles >= sms) {
        best_bt = bt;
        break;
      }
    }
    cudaError_t e;
    if (best_bt == 128)
      e = launch_router_tiled<Tx, 128>(c, x, w_router, logit_bias, logits, T, cfg.d, cfg.E);
    else if (best_bt == 64)
      e = launch_router_tiled<Tx, 64>(c, x, w_router, logit_bias, logits, T, cfg.d, cfg.E);
    else
      e = launch_router_tiled<Tx, 32>(c, x, w_router, logit_bias, logits, T, cfg.d, cfg.E);
    if (e != cudaSuccess) return e;
  }
  note_launches(1);
  return cudaGetLastError();
}

cudaError_t launch_router_logits(const Ctx& c, const moe_cfg& cfg, const void* x,
                                 const float* w_router, const float* logit_bias,
                                 float* logits, void* ws) {
  if (cfg.T > 0 && ws != nullptr && router_tc_eligible(cfg))
    return launch_router_logits_tc(c, cfg, x, w_router, logit_bias, logits, ws);
  if (cfg.act_dtype == MOE_BF16)
    return router_logits_dispatch(c, cfg, static_cast<const bf16*>(x), w_router, logit_bias,
                                  logits);
  return router_logits_dispatch(c, cfg, static_cast<const float*>(x), w_router, logit_bias,
                                logits);
}

static unsigned warp_grid(const Ctx& c, int64_t items) {
  const int64_t blocks = (items + 7) / 8;
  const int64_t cap = (int64_t)c.sm_count * 16;
  return (unsigned)(blocks < cap ? (blocks > 0 ? blocks : 1) : cap);
}

cudaError_t launch_router_topk(const Ctx& c, const moe_cfg& cfg, const float* logits,
                               const float* sel_bias, int32_t* idx, float* w) {
  return launch_router_topk_q(c, cfg, logits, sel_bias, nullptr, nullptr, idx, w);
}

cudaError_t launch_router_topk_q(const Ctx& c, const moe_cfg& cfg, const float* logits,
                                 const float* sel_bias, const float* beta, float* alpha,
                                 int32_t* idx, float* w) {
  if (cfg.T == 0) return cudaSuccess;
  const unsigned grid = warp_grid(c, cfg.T);
  const int epl = (cfg.E + 31) / 32;
  cudaError_t e;
  if (cfg.E <= 16) {
    // a group of 8 or 16 lanes per token
    if (cfg.E <= 8)
      e = launch_dependent(router_topk<1, 8>, dim3(warp_grid(c, (cfg.T + 3) / 4)), dim3(256), 0,
                           c.stream, logits, sel_bias, beta, alpha, idx, w, cfg.T, cfg.E, cfg.k,
                           cfg.score_fn, cfg.scaling);
    else
      e = launch_dependent(router_topk<1, 16>, dim3(warp_grid(c, (cfg.T + 1) / 2)), dim3(256), 0,
                           c.stream, logits, sel_bias, beta, alpha, idx, w, cfg.T, cfg.E, cfg.k,
                           cfg.score_fn, cfg.scaling);
    note_launches(1);
    return e;
  }
#define MOE_TOPK(N)                                                                          \
  e = launch_dependent(router_topk<N>, dim3(grid), dim3(256), 0, c.stream, logits, sel_bias, \
                       beta, alpha, idx, w, cfg.T, cfg.E, cfg.k, cfg.score_fn, cfg.scaling)
  switch (epl) {
    case 1: MOE_TOPK(1); break;
    case 2: MOE_TOPK(2); break;
    case 3: case 4: MOE_TOPK(4); break;
    default: MOE_TOPK(8); break;
  }
#undef MOE_TOPK
  note_launches(1);
  return e;
}

cudaError_t launch_router_near_ties(const Ctx& c, const moe_cfg& cfg, const float* logits,
                                    const float* sel_bias, float band, int32_t* count) {
  cudaError_t e = cudaMemsetAsync(count, 0, sizeof(int32_t), c.stream);
  if (e != cudaSuccess || cfg.T == 0 || cfg.k >= cfg.E) return e;
  const unsigned grid = warp_grid(c, cfg.T);
  const int epl = (cfg.E + 31) / 32;
#define MOE_TIES(N)                                                                   \
  router_near_ties<N><<<grid, 256, 0, c.stream>>>(logits, sel_bias, cfg.T, cfg.E, cfg.k, \
                                                  cfg.score_fn, band, count)
  switch (epl) {
    case 1: MOE_TIES(1); break;
    case 2: MOE_TIES(2); break;
    case 3: case 4: MOE_TIES(4); break;
    default: MOE_TIES(8); break;
  }
#undef MOE_TIES
  note_launches(1);
  return cudaGetLastError();
}

cudaError_t launch_router_scores_bwd(const Ctx& c, const moe_cfg& cfg, const float* logits,
                                     const int32_t* idx, const float* dw, float* d_logits,
                                     int accumulate) {
  if (cfg.T == 0) return cudaSuccess;
  if (cfg.E <= 16 && cfg.score_fn != MOE_SCORE_SOFTMAX_PRE) {
    const int64_t blocks = (cfg.T + 255) / 256;
    const int64_t cap = (int64_t)c.sm_count * 8;
    launch_dependent(router_scores_bwd_rows, dim3((unsigned)(blocks < cap ? blocks : cap)),
                     dim3(256), 0, c.stream, logits, idx, dw, d_logits, cfg.T, cfg.E, cfg.k,
                     cfg.score_fn, cfg.scaling, accumulate, c.status);
    note_launches(1);
    return cudaGetLastError();
  }
  launch_dependent(router_scores_bwd, dim3(warp_grid(c, cfg.T)), dim3(256), 0, c.stream,
      logits, idx, dw, d_logits, cfg.T, cfg.E, cfg.k, cfg.score_fn, cfg.scaling, accumulate,
      c.status);
  note_launches(1);
  return cudaGetLastError();
}

}  // namespace moe
