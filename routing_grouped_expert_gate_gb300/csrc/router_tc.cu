// Router gate GEMM (S1) on the tensor cores, at fp32 accuracy.
//
// The Ultimate MoE Training Handbook §3.1 "Router scoring", "Precision": the
// logits are l = x·W_rᵀ computed in fp32 from the [E, d] fp32 router weight;
// here x is the layer's bf16 activation.
//
// Method. Every fp32 weight is split exactly into three bf16 planes,
//   w0 = bf16(w),  w1 = bf16(w - w0),  w2 = bf16(w - w0 - w1),
// each subtraction exact in fp32; w - (w0 + w1 + w2) is below 2^-24 |w|.
// x is bf16, so every product x·wi is exact in fp32 and
//   x·W = x·W0 + x·W1 + x·W2
// loses nothing but the rounding of the fp32 sums. The x·W0 products carry
// the magnitude of the logit: they accumulate in TMEM over a short K window
// (fold_k elements) and the epilogue warps then fold the window's sum into a
// compensated (hi, lo) pair per logit (TwoSum), so the rounding that grows
// with d stays inside one window. The x·W1 and x·W2 products are 2^-8 and
// 2^-16 times smaller and accumulate over all of K in a 128-column TMEM
// accumulator (x·W1 beside x·W2: the two plane tiles sit back to back in
// shared memory, so one N = 128 MMA covers both); their rounding is far below
// fp32 resolution of the logit.
//
// One CTA computes 128 tokens x 64 experts: warp 0 issues the TMA loads (x
// tile + three W tiles per 64-wide K block); warp 1 owns 512 TMEM columns
// (six 64-column window accumulators, one 128-column low-part accumulator)
// and one of its lanes issues two tcgen05.mma per K16 step (M=128, K=16;
// N=64 for x·W0, N=128 for x·W1 | x·W2); warps 2..9 (two per TMEM lane
// quadrant, 32 columns each) fold the windows and write the logits, each fold
// thread keeping its token's 32 (hi, lo) pairs in registers; warp 10 waits on
// the mbarriers the MMA warp needs (the issuing thread never waits on an
// mbarrier). Every mbarrier wait is bounded (MOE_ERR_TIMEOUT + abort flag).
#include <algorithm>
#include <atomic>

#include "common.cuh"
#include "internal.h"
#include "tc_ptx.cuh"

namespace moe {
namespace rtc {

using namespace tc;

constexpr int R_EPI_WARPS = 8;  // fold warps: R_EPI_WARPS / 4 per TMEM lane quadrant
constexpr int R_RELAY_WARP = 2 + R_EPI_WARPS;  // waits for the MMA warp
constexpr int R_THREADS = 32 * (R_RELAY_WARP + 1);
constexpr int R_RELAY_BAR = 1;  // named barrier of the MMA and relay warps (64 threads)
constexpr int R_MAX_NWIN = 6;  // window accumulators in flight, at most
constexpr int R_MAX_STAGES = 8;

// TMEM columns for NW window accumulators of BN columns and the 2 BN
// low-part accumulator, rounded up to the power of two tcgen05.alloc takes.
constexpr int r_tmem_cols(int BN, int NW) {
  int c = 32;
  while (c < (NW + 2) * BN) c *= 2;
  return c;
}

// 32 lanes x 16 or 32 consecutive fp32 TMEM columns; the wait takes the
// registers as operands, so no use of them can move above it.
__device__ __forceinline__ void tmem_ld_cols(uint32_t taddr, float (&v)[32]) { tmem_ld32(taddr, v); }
__device__ __forceinline__ void tmem_ld_cols(uint32_t taddr, float (&v)[16]) {
  uint32_t r[16];
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 "
      "{%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15}, [%16];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
        "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]),
        "=r"(r[14]), "=r"(r[15])
      : "r"(taddr));
  asm volatile("tcgen05.wait::ld.sync.aligned;"
               : "+r"(r[0]), "+r"(r[1]), "+r"(r[2]), "+r"(r[3]), "+r"(r[4]), "+r"(r[5]),
                 "+r"(r[6]), "+r"(r[7]), "+r"(r[8]), "+r"(r[9]), "+r"(r[10]), "+r"(r[11]),
                 "+r"(r[12]), "+r"(r[13]), "+r"(r[14]), "+r"(r[15])
               :
               : "memory");
#pragma unroll
  for (int i = 0; i < 16; ++i) v[i] = __uint_as_float(r[i]);
}

template <int BN>
struct RTile {
  static constexpr int kA = 128 * 64 * 2;  // x: 128 tokens x 64 K, bf16
  static constexpr int kB = BN * 64 * 2;   // one W plane: BN experts x 64 K
  static constexpr int kStage = kA + 3 * kB;
  static constexpr int kStages = (200 * 1024) / kStage;  // 5 at BN = 64
  static_assert(kStages >= 2 && kStages <= R_MAX_STAGES, "pipeline depth");
};

struct RParams {
  int T, d, E;
  int fold;  // K16 steps per window of the x·W0 accumulator
  const float* logit_bias;
  float* logits;
  int* status;
  uint64_t timeout_ns;
};

struct __align__(8) RShared {
  uint64_t full[R_MAX_STAGES];
  uint64_t empty[R_MAX_STAGES];
  uint64_t acc_full[R_MAX_NWIN];
  uint64_t acc_empty[R_MAX_NWIN];
  uint64_t lo_full;
  uint32_t tmem_base;
  int abort;
};

template <int BN, int NW>
__global__ void __launch_bounds__(R_THREADS, 1)
router_logits_tc(const __grid_constant__ CUtensorMap tmX, const __grid_constant__ CUtensorMap tmW,
                 const RParams P) {
  using RT = RTile<BN>;
  constexpr int S = RT::kStages;
  constexpr int NC = BN / (R_EPI_WARPS / 4);  // columns per fold warp
  constexpr int CH = NC < 32 ? NC : 32;       // columns per TMEM read
  constexpr int COLS = r_tmem_cols(BN, NW);
  static_assert(NC % CH == 0 && (CH == 16 || CH == 32), "fold warp columns");
  static_assert(NW >= 2 && NW <= R_MAX_NWIN && COLS <= 512, "window accumulators");
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  RShared& sh = *reinterpret_cast<RShared*>(smem + S * RT::kStage);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int n0 = blockIdx.x * BN;   // first expert of the tile
  const int m0 = blockIdx.y * 128;  // first token of the tile
  const int nk = (P.d + 63) / 64;
  const int steps = nk * 4;  // K16 steps
  const int fold = P.fold;
  const int n_win = (steps + fold - 1) / fold;

  if (threadIdx.x == 0) {
    sh.abort = 0;
    for (int s = 0; s < S; ++s) {
      mbar_init(&sh.full[s], 1);
      mbar_init(&sh.empty[s], 1);
    }
    for (int a = 0; a < NW; ++a) {
      mbar_init(&sh.acc_full[a], 1);
      mbar_init(&sh.acc_empty[a], R_EPI_WARPS);  // one arrival per fold warp
    }
    mbar_init(&sh.lo_full, 1);
    fence_barrier_init();
  }
  if (warp == 1) {
    tmem_alloc(&sh.tmem_base, COLS);
    tmem_relinquish();
  }
  if (warp == 0 && lane == 0) {
    prefetch_tmap(&tmX);
    prefetch_tmap(&tmW);
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
      for (int kb = 0; kb < nk; ++kb) {
        if (!mbar_wait(&sh.empty[stage], phase ^ 1, sh.abort, P, 21)) { ok = false; break; }
        uint8_t* dst = smem + stage * RT::kStage;
        uint64_t* bar = &sh.full[stage];
        mbar_expect_tx(bar, RT::kStage);
        tma_load_2d(dst, &tmX, bar, kb * 64, m0);
#pragma unroll
        for (int p = 0; p < 3; ++p)
          tma_load_2d(dst + RT::kA + p * RT::kB, &tmW, bar, kb * 64, p * P.E + n0);
        if (++stage == S) { stage = 0; phase ^= 1; }
      }
      if (!ok) {
        // let the copies already in flight land before the CTA exits
        const uint64_t t0 = global_timer_ns();
        while (global_timer_ns() - t0 < 2000000ull) { }
      }
    }
  } else if (warp == 1) {
    // ================= MMA issuer =================
    // The whole warp walks the K16 steps in one flat loop and one lane issues:
    // at a step where the stage's tiles or the window's accumulator must be
    // waited for, the relay warp has done the waiting and the two warps meet
    // at R_RELAY_BAR (an mbarrier wait in the issuing thread stalls the tensor
    // pipe). The operand descriptors are the first stage's plus fixed offsets
    // (a stage is kStage bytes, a K16 step 32 bytes: 2 in the descriptor's
    // 16-byte units); at a stage's last step the stage is released to the
    // producer.
    constexpr uint32_t IDESC = idesc_bf16(false, false, 128, BN);
    constexpr uint32_t IDESC_LO = idesc_bf16(false, false, 128, 2 * BN);
    const uint32_t lo_acc = tmem + NW * BN;  // x·W1 in its first BN columns, x·W2 after
    const uint64_t d0 = sw128_desc(su32(smem), 16, 1024);
    int stage = 0;
    int pos = 0;  // the step's place in its window
    int buf = 0;  // the window's accumulator
    uint64_t da = d0;
    for (int step = 0; step < steps; ++step) {
      const int kk = step & 3;
      if (kk == 0 || pos == 0) {
        asm volatile("bar.sync %0, 64;" ::"r"(R_RELAY_BAR) : "memory");
        tc_fence_after();
      }
      if (kk == 0) da = d0 + (uint64_t)(stage * (RT::kStage >> 4));
      if (lane == 0) {
        const uint64_t a_d = da + (uint64_t)(2 * kk);
        const uint64_t b0_d = a_d + (uint64_t)(RT::kA >> 4);
        const uint64_t b1_d = b0_d + (uint64_t)(RT::kB >> 4);
        mma_bf16(tmem + buf * BN, a_d, b0_d, IDESC, pos > 0 ? 1u : 0u);
        mma_bf16(lo_acc, a_d, b1_d, IDESC_LO, step > 0 ? 1u : 0u);
      }
      if (++pos == fold || step == steps - 1) {
        if (lane == 0) mma_commit(&sh.acc_full[buf]);
        pos = 0;
        if (++buf == NW) buf = 0;
      }
      if (kk == 3) {
        if (lane == 0) mma_commit(&sh.empty[stage]);
        if (++stage == S) stage = 0;
      }
      __syncwarp();
    }
    if (lane == 0) mma_commit(&sh.lo_full);
    __syncwarp();
  } else if (warp == R_RELAY_WARP) {
    // ================= relay: the MMA warp's waits =================
    // After a failed wait (timeout or abort, recorded in the status word) it
    // stops waiting and only meets the MMA warp, which runs through its
    // remaining steps: no warp is left waiting.
    int stage = 0;
    uint32_t phase = 0;
    int pos = 0, buf = 0;
    uint32_t wphase = 0;
    bool ok = true;
    for (int step = 0; step < steps; ++step) {
      const int kk = step & 3;
      if (kk == 0 && ok) ok = mbar_wait(&sh.full[stage], phase, sh.abort, P, 22);
      // this buffer last held the window NW back: wait until it was folded
      if (pos == 0 && ok) ok = mbar_wait(&sh.acc_empty[buf], wphase ^ 1, sh.abort, P, 23);
      if (kk == 0 || pos == 0) asm volatile("bar.sync %0, 64;" ::"r"(R_RELAY_BAR) : "memory");
      if (++pos == fold || step == steps - 1) {
        pos = 0;
        if (++buf == NW) { buf = 0; wphase ^= 1; }
      }
      if (kk == 3 && ++stage == S) { stage = 0; phase ^= 1; }
    }
  } else {
    // ================= fold + store: warps 2..9 =================
    const int q = warp & 3;  // TMEM lanes 32q .. 32q+31 (the warp's quadrant)
    const int slice = (warp - 2) >> 2;  // the warp's NC of the tile's BN columns
    const int row = q * 32 + lane;
    const uint32_t base = tmem + ((uint32_t)(q * 32) << 16) + slice * NC;
    // Two levels: the window sums of a group of GROUP windows are added in
    // plain fp32 (round to nearest; the group's sum is a fraction of the
    // logit, so these roundings are far below the logit's ulp), and each
    // group sum folds into the compensated (hi, lo) pair with a TwoSum.
    constexpr int GROUP = 4;
    float hi[NC], lo[NC], grp[NC];
#pragma unroll
    for (int j = 0; j < NC; ++j) hi[j] = lo[j] = grp[j] = 0.f;
    bool ok = true;
    int buf = 0;
    uint32_t wphase = 0;
    for (int win = 0; win < n_win; ++win) {
      if (!mbar_wait(&sh.acc_full[buf], wphase, sh.abort, P, 24)) { ok = false; break; }
      tc_fence_after();
      const bool fold_now = (win % GROUP == GROUP - 1) || win == n_win - 1;
#pragma unroll
      for (int c = 0; c < NC; c += CH) {
        float v[CH];
        tmem_ld_cols(base + buf * BN + c, v);
        if (fold_now) {
#pragma unroll
          for (int i = 0; i < CH; ++i) {
            comp_add(hi[c + i], lo[c + i], __fadd_rn(grp[c + i], v[i]));
            grp[c + i] = 0.f;
          }
        } else {
#pragma unroll
          for (int i = 0; i < CH; ++i) grp[c + i] = __fadd_rn(grp[c + i], v[i]);
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&sh.acc_empty[buf]);
      if (++buf == NW) { buf = 0; wphase ^= 1; }
    }
    if (ok && mbar_wait(&sh.lo_full, 0, sh.abort, P, 25)) {
      tc_fence_after();
#pragma unroll
      for (int c = 0; c < NC; c += CH) {
#pragma unroll
        for (int p = 0; p < 2; ++p) {  // x·W1, then x·W2
          float v[CH];
          tmem_ld_cols(base + (NW + p) * BN + c, v);
#pragma unroll
          for (int i = 0; i < CH; ++i) lo[c + i] += v[i];
        }
      }
      const int64_t t = (int64_t)m0 + row;
      const int e0 = n0 + slice * NC;
      if (t < P.T) {
        float* dst = P.logits + t * P.E + e0;
#pragma unroll
        for (int j = 0; j < NC; j += 4) {
          float v[4];
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            float h = hi[j + i], l = lo[j + i];
            if (P.logit_bias != nullptr) comp_add(h, l, P.logit_bias[e0 + j + i]);
            v[i] = __fadd_rn(h, l);
          }
          *reinterpret_cast<float4*>(dst + j) = make_float4(v[0], v[1], v[2], v[3]);
        }
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, COLS);
  }
}

// w [n] fp32 -> planes [3][n] bf16 with w = p0 + p1 + p2 (to 2^-24 |w|)
__global__ void router_split_planes(const float* __restrict__ w, bf16* __restrict__ planes,
                                    int64_t n4) {
  pdl_wait();  // a dependent launch: inputs come from the kernels before
  const int64_t n = 4 * n4;
  for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < n4;
       i += (int64_t)gridDim.x * blockDim.x) {
    const float4 v4 = reinterpret_cast<const float4*>(w)[i];
    const float v[4] = {v4.x, v4.y, v4.z, v4.w};
    bf16 p0[4], p1[4], p2[4];
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      p0[j] = __float2bfloat16_rn(v[j]);
      const float r1 = v[j] - __bfloat162float(p0[j]);  // exact
      p1[j] = __float2bfloat16_rn(r1);
      const float r2 = r1 - __bfloat162float(p1[j]);  // exact
      p2[j] = __float2bfloat16_rn(r2);
    }
    *reinterpret_cast<uint2*>(planes + 4 * i) = *reinterpret_cast<const uint2*>(p0);
    *reinterpret_cast<uint2*>(planes + n + 4 * i) = *reinterpret_cast<const uint2*>(p1);
    *reinterpret_cast<uint2*>(planes + 2 * n + 4 * i) = *reinterpret_cast<const uint2*>(p2);
  }
}

template <int BN>
constexpr size_t r_smem_bytes() {
  return 1024 + (size_t)RTile<BN>::kStages * RTile<BN>::kStage + sizeof(RShared);
}

template <int BN, int NW>
static cudaError_t launch_tc(const Ctx& c, const CUtensorMap& mx, const CUtensorMap& mw,
                             const RParams& P) {
  auto kern = router_logits_tc<BN, NW>;
  constexpr size_t smem = r_smem_bytes<BN>();
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
  dim3 grid((unsigned)(P.E / BN), (unsigned)((P.T + 127) / 128));
  kern<<<grid, R_THREADS, smem, c.stream>>>(mx, mw, P);
  return cudaGetLastError();
}

static std::atomic<int> g_router_impl{0};   // 0: tensor cores where eligible; 1: CUDA cores
static std::atomic<int> g_router_fold{32};  // K elements per window of the x·W0 accumulator

}  // namespace rtc

bool router_tc_eligible(const moe_cfg& cfg) {
  return cfg.act_dtype == MOE_BF16 && cfg.E >= 64 && cfg.E % 64 == 0 && cfg.d >= 64 &&
         cfg.T <= (int64_t)65535 * 128 &&  // token tiles ride on gridDim.y
         rtc::g_router_impl.load() == 0 && tc_available();
}

size_t router_ws_bytes(const moe_cfg& cfg) {
  if (cfg.act_dtype != MOE_BF16 || cfg.E < 64 || cfg.E % 64 != 0 || cfg.d < 64) return 0;
  return ((size_t)3 * cfg.E * cfg.d * sizeof(bf16) + 255) & ~(size_t)255;
}

int router_set_impl(int impl) { return rtc::g_router_impl.exchange(impl); }

bool router_tensor_cores_enabled() { return rtc::g_router_impl.load() == 0; }

int router_set_fold(int fold_k) { return rtc::g_router_fold.exchange(fold_k); }

cudaError_t launch_router_logits_tc(const Ctx& c, const moe_cfg& cfg, const void* x,
                                    const float* w_router, const float* logit_bias,
                                    float* logits, void* ws) {
  using namespace rtc;
  const int64_t n = (int64_t)cfg.E * cfg.d;
  bf16* planes = static_cast<bf16*>(ws);
  const int64_t n4 = n / 4;
  const int blocks = (int)std::min<int64_t>((n4 + 255) / 256, (int64_t)c.sm_count * 8);
  launch_dependent(router_split_planes, dim3(blocks), dim3(256), 0, c.stream, w_router, planes, n4);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  note_launches(1);

  constexpr int BN = 64;
  CUtensorMap mx, mw;
  if (!tc::make_map_bf16(&mx, x, cfg.T, cfg.d, 128) ||
      !tc::make_map_bf16(&mw, planes, 3 * (int64_t)cfg.E, cfg.d, BN))
    return cudaErrorInvalidValue;
  RParams P{};
  P.T = (int)cfg.T;
  P.d = cfg.d;
  P.E = cfg.E;
  P.fold = std::max(1, g_router_fold.load() / 16);
  P.logit_bias = logit_bias;
  P.logits = logits;
  P.status = c.status;
  P.timeout_ns = c.timeout_ns;
  e = launch_tc<BN, 6>(c, mx, mw, P);
  note_launches(1);
  return e;
}

}  // namespace moe
