// Router backward GEMMs (B1/B3) on the tensor cores, at fp32 accuracy.
//
// The Ultimate MoE Training Handbook §3.1 "Router scoring", "Precision": the
// router runs in fp32. Its backward has two products of the fp32 logit
// gradient G = d_logits [T, E]:
//   dx_router = G · W_r   [T, d]   (K = E)
//   dW_r      = Gᵀ · x    [E, d]   (K = T, split into slices summed in order)
// Both run as sums of bf16 products of exact planes: G = G0 + G1 + G2 and
// W_r = W0 + W1 + W2 (each plane the bf16 rounding of what the planes before
// it leave over). dx_router keeps the six products whose combined scale is
// at least 2^-16 of the leading one (G0W0, G0W1, G1W0, G0W2, G1W1, G2W0); the
// dropped ones are below 2^-24 relative. dW_r needs three (x is bf16, exact):
// G0x, G1x, G2x. Every product is exact in fp32 and accumulates in TMEM.
//
// One persistent kernel template computes C[M, N] (fp32) = Σ_pairs A_p · B_q
// over a K range, 128 x BNT tiles: warp 0 issues TMA loads of the planes per
// 64-wide K block, warp 1 owns TMEM (two accumulators) and issues
// tcgen05.mma (M=128, N=BNT, K=16) for every plane pair, warps 2..9 drain the
// idle accumulator (two warps per lane quadrant) with 16-byte fp32 stores,
// warp 10 waits on the mbarriers the MMA warp needs (a named barrier per
// stage between the two: the issuing thread never waits on an mbarrier).
// Split K writes slice partials [S][M][N], summed afterwards in slice order.
// Every mbarrier wait is bounded (MOE_ERR_TIMEOUT + abort flag).
#include <algorithm>
#include <atomic>

#include "common.cuh"
#include "internal.h"
#include "tc_ptx.cuh"

namespace moe {
namespace rbw {

using namespace tc;

constexpr int PB_EPI_WARPS = 8;
constexpr int PB_RELAY_WARP = 2 + PB_EPI_WARPS;  // waits for the MMA warp
constexpr int PB_THREADS = 32 * (PB_RELAY_WARP + 1);
constexpr int PB_RELAY_BAR = 1;  // named barrier of the MMA and relay warps (64 threads)
constexpr int PB_MAX_STAGES = 4;

struct PParams {
  int M, N, K;            // C is [M, N]; A planes [3][M or K ...] per the tensor maps
  int k_per_split, splits;
  int a_plane_rows;       // rows of one A plane in its tensor map (K-major: M; MN-major: K)
  int b_plane_rows;       // rows of one B plane (K-major: N; MN-major: K)
  int m_tiles, n_tiles;
  float* out;             // [splits][M][N] fp32
  int* status;
  uint64_t timeout_ns;
};

struct __align__(8) PShared {
  uint64_t full[PB_MAX_STAGES];
  uint64_t empty[PB_MAX_STAGES];
  uint64_t acc_full[2];
  uint64_t acc_empty[2];
  uint32_t tmem_base;
  int abort;
};

// NP plane pairs: (pa[j], pb[j])
template <int NP>
struct Pairs;
template <>
struct Pairs<6> {
  static constexpr int NA = 3, NB = 3;
  __device__ static int a(int j) { return j == 0 || j == 1 || j == 3 ? 0 : (j == 2 || j == 4 ? 1 : 2); }
  __device__ static int b(int j) { return j == 0 || j == 2 || j == 5 ? 0 : (j == 1 || j == 4 ? 1 : 2); }
};
template <>
struct Pairs<3> {
  static constexpr int NA = 3, NB = 1;
  __device__ static int a(int j) { return j; }
  __device__ static int b(int) { return 0; }
};

template <int NP, int BNT>
struct PTile {
  static constexpr int kA = 128 * 64 * 2;   // one A plane: 128 M x 64 K
  static constexpr int kB = BNT * 64 * 2;   // one B plane: BNT N x 64 K
  static constexpr int kStage = Pairs<NP>::NA * kA + Pairs<NP>::NB * kB;
  static constexpr int kStages = (200 * 1024) / kStage;
  static_assert(kStages >= 2 && kStages <= PB_MAX_STAGES, "pipeline depth");
};

struct PTileId {
  int m0, n0, split, k0, nk;
};

__device__ __forceinline__ PTileId decode(const PParams& P, int t) {
  PTileId id;
  const int per = P.m_tiles * P.n_tiles;
  id.split = t / per;
  const int r = t - id.split * per;
  const int mi = r / P.n_tiles;
  id.n0 = (r - mi * P.n_tiles);
  id.m0 = mi * 128;
  id.k0 = id.split * P.k_per_split;
  int k1 = id.k0 + P.k_per_split;
  if (k1 > P.K) k1 = P.K;
  id.nk = k1 > id.k0 ? (k1 - id.k0 + 63) / 64 : 0;
  return id;
}

template <bool A_MN, bool B_MN, int NP, int BNT>
__global__ void __launch_bounds__(PB_THREADS, 1)
plane_gemm(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
           const PParams P) {
  using PT = PTile<NP, BNT>;
  using PR = Pairs<NP>;
  constexpr int S = PT::kStages;
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  PShared& sh = *reinterpret_cast<PShared*>(smem + S * PT::kStage);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int total = P.m_tiles * P.n_tiles * P.splits;

  if (threadIdx.x == 0) {
    sh.abort = 0;
    for (int s = 0; s < S; ++s) {
      mbar_init(&sh.full[s], 1);
      mbar_init(&sh.empty[s], 1);
    }
    for (int a = 0; a < 2; ++a) {
      mbar_init(&sh.acc_full[a], 1);
      mbar_init(&sh.acc_empty[a], PB_EPI_WARPS);  // one arrival per epilogue warp
    }
    fence_barrier_init();
  }
  if (warp == 1) {
    tmem_alloc(&sh.tmem_base, 2 * BNT);
    tmem_relinquish();
  }
  if (warp == 0 && lane == 0) {
    prefetch_tmap(&tmA);
    prefetch_tmap(&tmB);
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = sh.tmem_base;

  if (warp == 0) {
    // ================= TMA producer =================
    if (lane == 0) {
      int stage = 0;
      uint32_t phase = 0;
      bool ok = true;
      for (int t = blockIdx.x; t < total && ok; t += gridDim.x) {
        const PTileId id = decode(P, t);
        const int n0 = id.n0 * BNT;
        for (int kb = 0; kb < id.nk; ++kb) {
          if (!mbar_wait(&sh.empty[stage], phase ^ 1, sh.abort, P, 31)) { ok = false; break; }
          uint8_t* dst = smem + stage * PT::kStage;
          uint64_t* bar = &sh.full[stage];
          mbar_expect_tx(bar, PT::kStage);
          const int k = id.k0 + kb * 64;
#pragma unroll
          for (int p = 0; p < PR::NA; ++p) {
            uint8_t* a_dst = dst + p * PT::kA;
            if (!A_MN) {
              tma_load_2d(a_dst, &tmA, bar, k, p * P.a_plane_rows + id.m0);
            } else {
              tma_load_2d(a_dst, &tmA, bar, id.m0, p * P.a_plane_rows + k);
              tma_load_2d(a_dst + 8192, &tmA, bar, id.m0 + 64, p * P.a_plane_rows + k);
            }
          }
#pragma unroll
          for (int q = 0; q < PR::NB; ++q) {
            uint8_t* b_dst = dst + PR::NA * PT::kA + q * PT::kB;
            if (!B_MN) {
              tma_load_2d(b_dst, &tmB, bar, k, q * P.b_plane_rows + n0);
            } else {
#pragma unroll
              for (int j = 0; j < BNT / 64; ++j)
                tma_load_2d(b_dst + j * 8192, &tmB, bar, n0 + 64 * j, q * P.b_plane_rows + k);
            }
          }
          if (++stage == S) { stage = 0; phase ^= 1; }
        }
      }
      if (!ok) {
        const uint64_t t0 = global_timer_ns();
        while (global_timer_ns() - t0 < 2000000ull) { }
      }
    }
  } else if (warp == 1) {
    // ================= MMA issuer =================
    constexpr uint32_t IDESC = idesc_bf16(A_MN, B_MN, 128, BNT);
    int stage = 0, acc = 0;
    for (int t = blockIdx.x; t < total; t += gridDim.x) {
      const PTileId id = decode(P, t);
      if (id.nk == 0) continue;  // an empty K slice: the epilogue writes its zeros itself
      const uint32_t d_tmem = tmem + acc * BNT;
      for (int kb = 0; kb < id.nk; ++kb) {
        // the relay warp has seen this stage's tiles land (and, at kb == 0,
        // this accumulator drained): an mbarrier wait in the issuing thread
        // stalls the tensor pipe, a named barrier does not
        asm volatile("bar.sync %0, 64;" ::"r"(PB_RELAY_BAR) : "memory");
        tc_fence_after();
        if (lane == 0) {
          const uint32_t base = su32(smem + stage * PT::kStage);
#pragma unroll
          for (int kk = 0; kk < 4; ++kk) {
#pragma unroll
            for (int j = 0; j < NP; ++j) {
              const uint32_t a_addr = base + PR::a(j) * PT::kA;
              const uint32_t b_addr = base + PR::NA * PT::kA + PR::b(j) * PT::kB;
              const uint64_t ad = !A_MN ? sw128_desc(a_addr + kk * 32, 16, 1024)
                                        : sw128_desc(a_addr + kk * 2048, 8192, 1024);
              const uint64_t bd = !B_MN ? sw128_desc(b_addr + kk * 32, 16, 1024)
                                        : sw128_desc(b_addr + kk * 2048, 8192, 1024);
              mma_bf16(d_tmem, ad, bd, IDESC, (kb | kk | j) != 0 ? 1u : 0u);
            }
          }
          mma_commit(&sh.empty[stage]);
        }
        __syncwarp();
        if (++stage == S) stage = 0;
      }
      if (lane == 0) mma_commit(&sh.acc_full[acc]);
      __syncwarp();
      acc ^= 1;
    }
  } else if (warp == PB_RELAY_WARP) {
    // ================= relay: the MMA warp's waits =================
    // After a failed wait (timeout or abort, recorded in the status word) it
    // stops waiting and only meets the MMA warp, which runs through its
    // remaining k-blocks: no warp is left waiting.
    int stage = 0, acc = 0;
    uint32_t phase = 0, acc_phase = 0;
    bool ok = true;
    for (int t = blockIdx.x; t < total; t += gridDim.x) {
      const PTileId id = decode(P, t);
      if (id.nk == 0) continue;
      for (int kb = 0; kb < id.nk; ++kb) {
        if (ok && kb == 0) ok = mbar_wait(&sh.acc_empty[acc], acc_phase ^ 1, sh.abort, P, 32);
        if (ok) ok = mbar_wait(&sh.full[stage], phase, sh.abort, P, 33);
        asm volatile("bar.sync %0, 64;" ::"r"(PB_RELAY_BAR) : "memory");
        if (++stage == S) { stage = 0; phase ^= 1; }
      }
      acc ^= 1;
      if (acc == 0) acc_phase ^= 1;
    }
  } else {
    // ================= epilogue: warps 2..9 =================
    const int q = warp & 3, half = (warp - 2) >> 2;
    const int row = q * 32 + lane;
    int acc = 0;
    uint32_t acc_phase = 0;
    for (int t = blockIdx.x; t < total; t += gridDim.x) {
      const PTileId id = decode(P, t);
      const int m = id.m0 + row;
      const int n0 = id.n0 * BNT;
      float* dst = P.out + (int64_t)id.split * P.M * P.N + (int64_t)m * P.N;
      if (id.nk == 0) {  // an empty K slice: its partial is zero
        if (m < P.M)
          for (int c = half * (BNT / 2); c < (half + 1) * (BNT / 2); c += 4)
            if (n0 + c < P.N) *reinterpret_cast<float4*>(dst + n0 + c) = make_float4(0, 0, 0, 0);
        continue;
      }
      if (!mbar_wait(&sh.acc_full[acc], acc_phase, sh.abort, P, 34)) break;
      tc_fence_after();
      const uint32_t t_row = tmem + ((uint32_t)(q * 32) << 16) + acc * BNT;
#pragma unroll 1
      for (int c = half * (BNT / 2); c < (half + 1) * (BNT / 2); c += 32) {
        float v[32];
        tmem_ld32(t_row + c, v);
        if (m < P.M) {
#pragma unroll
          for (int j = 0; j < 8; ++j)
            if (n0 + c + 4 * j < P.N)
              *reinterpret_cast<float4*>(dst + n0 + c + 4 * j) =
                  make_float4(v[4 * j], v[4 * j + 1], v[4 * j + 2], v[4 * j + 3]);
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&sh.acc_empty[acc]);
      acc ^= 1;
      if (acc == 0) acc_phase ^= 1;
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, 2 * BNT);
  }
}

// fp32 [n] -> three bf16 planes [3][n] (the same split as the forward's)
__global__ void split3(const float* __restrict__ v, bf16* __restrict__ planes, int64_t n4) {
  pdl_wait();  // a dependent launch: inputs come from the kernels before
  const int64_t n = 4 * n4;
  for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < n4;
       i += (int64_t)gridDim.x * blockDim.x) {
    const float4 x4 = reinterpret_cast<const float4*>(v)[i];
    const float xs[4] = {x4.x, x4.y, x4.z, x4.w};
    bf16 p0[4], p1[4], p2[4];
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      p0[j] = __float2bfloat16_rn(xs[j]);
      const float r1 = xs[j] - __bfloat162float(p0[j]);
      p1[j] = __float2bfloat16_rn(r1);
      p2[j] = __float2bfloat16_rn(r1 - __bfloat162float(p1[j]));
    }
    *reinterpret_cast<uint2*>(planes + 4 * i) = *reinterpret_cast<const uint2*>(p0);
    *reinterpret_cast<uint2*>(planes + n + 4 * i) = *reinterpret_cast<const uint2*>(p1);
    *reinterpret_cast<uint2*>(planes + 2 * n + 4 * i) = *reinterpret_cast<const uint2*>(p2);
  }
}

template <bool A_MN, bool B_MN, int NP, int BNT>
static cudaError_t launch_plane_gemm(const Ctx& c, const CUtensorMap& ma, const CUtensorMap& mb,
                                     const PParams& P) {
  using PT = PTile<NP, BNT>;
  auto kern = plane_gemm<A_MN, B_MN, NP, BNT>;
  constexpr size_t smem = 1024 + (size_t)PT::kStages * PT::kStage + sizeof(PShared);
  static std::atomic<uint64_t> attr_set_mask{0};
  int dev = 0;
  cudaGetDevice(&dev);
  const uint64_t bit = 1ull << (dev & 63);
  if (!(attr_set_mask.load() & bit)) {
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)smem);
    if (e != cudaSuccess) return e;
    attr_set_mask.fetch_or(bit);
  }
  const int total = P.m_tiles * P.n_tiles * P.splits;
  const int grid = std::max(1, std::min(total, c.sm_count));
  kern<<<grid, PB_THREADS, smem, c.stream>>>(ma, mb, P);
  note_launches(1);
  return cudaGetLastError();
}

static void split_planes(const Ctx& c, const float* v, bf16* planes, int64_t n) {
  const int64_t n4 = n / 4;
  const int blocks = (int)std::max<int64_t>(1, std::min<int64_t>((n4 + 255) / 256,
                                                                 (int64_t)c.sm_count * 8));
  launch_dependent(split3, dim3(blocks), dim3(256), 0, c.stream, v, planes, n4);
  note_launches(1);
}

}  // namespace rbw

// Workspace: G planes [3][T][E] bf16, W planes [3][E][d] bf16, dW slice partials
// [S][E][d] fp32. S: enough (E-tile x d-tile x slice) tiles for every SM.
// (a fixed target of 304 CTAs keeps the workspace size independent of the device)
static int router_bwd_tc_splits(const moe_cfg& cfg) {
  const int64_t tiles = ((cfg.E + 127) / 128) * ((cfg.d + 255) / 256);
  int64_t s = (304 + tiles - 1) / tiles;
  const int64_t max_s = (cfg.T + 255) / 256;  // at least 256 tokens per slice
  if (s > max_s) s = max_s;
  if (s < 1) s = 1;
  return (int)s;
}

bool router_bwd_tc_shape(const moe_cfg& cfg) {
  return cfg.act_dtype == MOE_BF16 && cfg.E >= 32 && cfg.E % 8 == 0 &&
         3 * cfg.T <= (int64_t)0x7fffffff;
}

bool router_bwd_tc_eligible(const moe_cfg& cfg) {
  return router_bwd_tc_shape(cfg) && router_tensor_cores_enabled() && tc_available();
}

size_t router_bwd_tc_ws_bytes(const moe_cfg& cfg) {
  auto r256 = [](size_t n) { return (n + 255) & ~(size_t)255; };
  const int S = router_bwd_tc_splits(cfg);
  return r256((size_t)3 * cfg.T * cfg.E * 2) + r256((size_t)3 * cfg.E * cfg.d * 2) +
         r256((size_t)S * cfg.E * cfg.d * 4);
}

cudaError_t launch_router_bwd_tc(const Ctx& c, const moe_cfg& cfg, const void* x,
                                 const float* w_router, const float* d_logits, float* dx_router,
                                 float* dw_router, void* ws) {
  using namespace rbw;
  auto r256 = [](size_t n) { return (n + 255) & ~(size_t)255; };
  const int64_t T = cfg.T;
  const int E = cfg.E, d = cfg.d;
  uint8_t* base = static_cast<uint8_t*>(ws);
  bf16* gp = reinterpret_cast<bf16*>(base);
  base += r256((size_t)3 * T * E * 2);
  bf16* wp = reinterpret_cast<bf16*>(base);
  base += r256((size_t)3 * E * d * 2);
  float* part = reinterpret_cast<float*>(base);
  split_planes(c, d_logits, gp, T * E);
  split_planes(c, w_router, wp, (int64_t)E * d);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;

  // dx_router [T, d] = Σ Gp · Wq: A = G planes K-major ([3T, E], box 64 x 128),
  // B = W planes MN-major ([3E, d], boxes 64 x 64), 128-column tiles, 6 pairs
  {
    CUtensorMap ma, mb;
    if (!tc::make_map_bf16(&ma, gp, 3 * T, E, 128) || !tc::make_map_bf16(&mb, wp, 3 * (int64_t)E, d, 64))
      return cudaErrorInvalidValue;
    PParams P{};
    P.M = (int)T; P.N = d; P.K = E;
    P.k_per_split = E; P.splits = 1;
    P.a_plane_rows = (int)T; P.b_plane_rows = E;
    P.m_tiles = (int)((T + 127) / 128); P.n_tiles = (d + 127) / 128;
    P.out = dx_router;
    P.status = c.status; P.timeout_ns = c.timeout_ns;
    e = launch_plane_gemm<false, true, 6, 128>(c, ma, mb, P);
    if (e != cudaSuccess) return e;
  }
  // dW_r [E, d] = Σ Gpᵀ · x: A = G planes MN-major ([3T, E], boxes 64 x 64),
  // B = x MN-major ([T, d], boxes 64 x 64), 256-column tiles, 3 pairs, K = T in slices
  {
    const int S = router_bwd_tc_splits(cfg);
    CUtensorMap ma, mb;
    if (!tc::make_map_bf16(&ma, gp, 3 * T, E, 64) || !tc::make_map_bf16(&mb, x, T, d, 64))
      return cudaErrorInvalidValue;
    PParams P{};
    P.M = E; P.N = d; P.K = (int)T;
    P.k_per_split = (int)(((T + S - 1) / S + 63) / 64 * 64); P.splits = S;
    P.a_plane_rows = (int)T; P.b_plane_rows = (int)T;
    P.m_tiles = (E + 127) / 128; P.n_tiles = (d + 255) / 256;
    P.out = part;
    P.status = c.status; P.timeout_ns = c.timeout_ns;
    e = launch_plane_gemm<true, true, 3, 256>(c, ma, mb, P);
    if (e != cudaSuccess) return e;
    e = launch_reduce_partials(c, part, (int64_t)E * d, S, (int64_t)E * d, dw_router, kF32, 0);
  }
  return e;
}

}  // namespace moe
