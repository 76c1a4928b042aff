// Grouped expert GEMMs on the 5th-generation tensor cores (tcgen05 + TMEM + TMA).
//
// The Ultimate MoE Training Handbook, §3.4 "Experts": each expert is a bias-free
// SwiGLU FFN whose fc1 is 2F wide (gate half first, "Activation") and whose fc2
// maps F back to d ("Count and size"); the local experts' GEMMs run as one
// grouped GEMM. MoE training cluster: routing, load balancing (LeCompute),
// "Read the timeline before blaming the network": grouping lets a GPU stay busy
// even when single experts receive few tokens.
//
// One persistent, warp-specialised kernel template serves every contraction of
// the layer's expert FFNs (bf16 operands, fp32 accumulation in TMEM):
//
//   fc1 forward    h = silu(x W1gᵀ) * (x W1uᵀ)   M-grouped, SwiGLU epilogue
//   fc2 forward    out = h W2ᵀ                    M-grouped
//   fc2 dgrad      d_pre = SwiGLU'(d_out W2)      M-grouped, SwiGLU-backward epilogue
//   fc1 dgrad      dx = d_pre W1                  M-grouped
//   fc2 wgrad      dW2_e = d_outᵀ h               K-grouped (K = the expert's rows)
//   fc1 wgrad      dW1_e = d_preᵀ x               K-grouped
//
// Tiles are 128 x 256 (M x N) with K stepping 64 bf16 (one 128-byte swizzle row)
// per pipeline stage. Warp 0 issues TMA loads into a 4-stage shared-memory ring;
// warp 1 allocates 512 TMEM columns (two 256-column fp32 accumulators) and one
// of its threads issues tcgen05.mma (M=128, N=256, K=16); warps 2..9 drain an
// accumulator through tcgen05.ld while the next tile accumulates in the other;
// warp 10 waits on the mbarriers the MMA warp needs and meets it at a named
// barrier per stage, so that the issuing thread never waits on an mbarrier.
// The tile list is built on the device from the segment offsets: no host sync.
// M-grouped tiles of one expert run m-fastest so that concurrently running CTAs
// share the expert's weight tile through L2. K-grouped tiles take the experts
// longest-first.
//
// Safety: every mbarrier wait is bounded by the caller's timeout (globaltimer);
// on expiry the kernel records MOE_ERR_TIMEOUT, raises an abort flag that every
// role polls, waits (bounded) for its own TMA copies, frees TMEM and returns.
#include <cuda.h>
#include <cudaTypedefs.h>

#include <atomic>
#include <mutex>
#include <vector>

#include "common.cuh"
#include "internal.h"
#include "glu_act.cuh"
#include "tc_ptx.cuh"

namespace moe {
namespace tc {

constexpr int BM = 128;
constexpr int BN = 256;
constexpr int BK = 64;
constexpr int STAGES = 4;
constexpr int A_STAGE_BYTES = BM * BK * 2;      // 16 KB
constexpr int B_STAGE_BYTES = BN * BK * 2;      // 32 KB
constexpr int STAGE_BYTES = A_STAGE_BYTES + B_STAGE_BYTES;
constexpr int NUM_EPI_WARPS = 8;                 // two per TMEM lane quadrant
constexpr int RELAY_WARP = 2 + NUM_EPI_WARPS;     // waits for the MMA warp (after the epilogue warps)
constexpr int NUM_THREADS = 32 * (RELAY_WARP + 1);  // producer, MMA, epilogue, relay warps
constexpr int RELAY_BAR = 1;                      // named barrier of the MMA and relay warps
constexpr int TMEM_COLS = 512;
constexpr int MAXG = 256;
// per epilogue warp: one 32 x 32 bf16 output box staged for a TMA store
constexpr int EPI_BOX_BYTES = 32 * 32 * 2;
constexpr int EPI_BUF_BYTES = NUM_EPI_WARPS * EPI_BOX_BYTES;  // 16 KB

enum Epi { EPI_STORE = 0, EPI_SWIGLU_FWD = 1, EPI_SWIGLU_BWD = 2, EPI_WGRAD = 3 };

struct Params {
  int G;              // groups (experts)
  int n_rows;         // rows of the grouped operand (sum of the segments)
  int K;              // M-grouped: reduction length
  int N_out;          // output columns (M-grouped) / per-group N (K-grouped)
  int M_out;          // K-grouped: per-group M
  int NT, MT;         // tiles along N (and M for K-grouped)
  int b_group_rows;   // M-grouped: rows of the B tensor map per group
  int F;              // SwiGLU width
  const int32_t* offsets;  // [G+1], NULL = one group of n_rows
  bf16* out0;
  int64_t ld0;
  bf16* out1;         // fc1 forward: gate|up output (may be NULL)
  const bf16* aux_in; // fc2 dgrad: gate|up input
  int* status;
  uint64_t timeout_ns;
  GluAct act;         // expert activation (SwiGLU epilogues)
  int tma_out;        // 1: outputs leave as staged boxes (TMA stores; the weight
                      //    gradients' through the warps' own stores), 0: per thread
  // K-grouped: per group, the A map with its rows ending at the group's last
  // row (rows after it read as zeros), for the group's last K block; NULL =
  // the MMA warp zeroes those rows in shared memory instead
  const CUtensorMap* tail_maps;
  int m128_tails;     // CTA pairs, M-grouped: a last tile of <= 128 rows runs as M = 128
  // gathered A (fc1 forward): row r of the A operand is row a_src[r] of a_rows
  // [a_src_rows, K]; rows r >= n_rows read as zeros
  const bf16* a_rows;
  const int32_t* a_src;
  int a_src_rows;
};

struct __align__(8) Shared {
  uint64_t full[STAGES];
  uint64_t empty[STAGES];
  uint64_t tmem_full[2];
  uint64_t tmem_empty[2];
  uint64_t epi_load[NUM_EPI_WARPS];  // TMA loads into an epilogue warp's buffer
  uint32_t tmem_base;
  int abort;
  int total_tiles;
  int off[MAXG + 1];
  int prefix[MAXG + 1];
  int order[MAXG];
};

// Named barrier of two whole warps (64 threads): the MMA warp and its relay.
__device__ __forceinline__ void warp_pair_sync(int id) {
  asm volatile("bar.sync %0, 64;" ::"r"(id) : "memory");
}

// The relay warp: it walks the MMA warp's tiles and k-blocks, waits on the
// barriers the MMA warp needs (at a tile's first k-block the accumulator's
// tmem_empty, then the stage's full) and meets the MMA warp at RELAY_BAR once
// per k-block. An mbarrier wait in the thread that issues the MMAs stalls the
// tensor pipe at every stage (measured: 4 N=256 MMAs per stage take 512
// cycles from one thread alone, 670 with a wait on an already completed
// barrier and a commit per stage, 512 with the wait moved to this warp); the
// named barrier costs nothing there. After a failed wait (timeout or abort,
// recorded in the status word) the relay stops waiting and only meets the
// MMA warp, which runs through its remaining k-blocks on whatever the stages
// hold: the call reports the error, and no warp is left waiting.
template <class SH, class PP, class Decode>
__device__ __forceinline__ void relay_waits(SH& sh, const PP& P, int t0, int tstep, int total,
                                            Decode decode, int stages, int accs, int site) {
  int stage = 0, acc = 0;
  uint32_t phase = 0, acc_phase = 0;
  bool ok = true;
  for (int t = t0; t < total; t += tstep) {
    const auto ti = decode(t);
    if (ti.nk == 0) continue;
    for (int kb = 0; kb < ti.nk; ++kb) {
      if (ok && kb == 0) ok = mbar_wait(&sh.tmem_empty[acc], acc_phase ^ 1, sh.abort, P, site);
      if (ok) ok = mbar_wait(&sh.full[stage], phase, sh.abort, P, site + 1);
      warp_pair_sync(RELAY_BAR);
      if (++stage == stages) { stage = 0; phase ^= 1; }
    }
    if (++acc == accs) { acc = 0; acc_phase ^= 1; }
  }
}

// Instruction descriptor of kind::f16: fp32 accumulator, bf16 A and B,
// A/B major-ness (0 = K-major, 1 = MN-major), N>>3 at [17,23), M>>4 at [24,29).
__host__ __device__ constexpr uint32_t make_idesc(bool a_mn, bool b_mn) {
  return (1u << 4) | (1u << 7) | (1u << 10) | ((a_mn ? 1u : 0u) << 15) |
         ((b_mn ? 1u : 0u) << 16) | ((uint32_t)(BN >> 3) << 17) | ((uint32_t)(BM >> 4) << 24);
}

__device__ __forceinline__ float silu_f(float g) { return g / (1.f + __expf(-g)); }

__device__ __forceinline__ void store_bf16x8(bf16* p, const float* v) {
  uint4 r;
  __nv_bfloat162* h = reinterpret_cast<__nv_bfloat162*>(&r);
#pragma unroll
  for (int i = 0; i < 4; ++i) h[i] = __floats2bfloat162_rn(v[2 * i], v[2 * i + 1]);
  *reinterpret_cast<uint4*>(p) = r;
}
__device__ __forceinline__ void load_bf16x8(const bf16* p, float* v) {
  uint4 r = *reinterpret_cast<const uint4*>(p);
  const __nv_bfloat162* h = reinterpret_cast<const __nv_bfloat162*>(&r);
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    float2 f = __bfloat1622float2(h[i]);
    v[2 * i] = f.x;
    v[2 * i + 1] = f.y;
  }
}

// One row (thread = lane = row) of a 32 x 32 bf16 box into the warp's staging
// buffer, laid out as the output tensor map's 64-byte swizzle expects: the
// 16-byte chunk j of row r sits at chunk j ^ ((r >> 1) & 3) of the row's 64
// bytes. Eight consecutive rows then cover all 32 banks, so the warp's 16-byte
// stores are free of bank conflicts. The buffer is 1024-byte aligned.
__device__ __forceinline__ void stage_box_row(uint32_t buf, int lane, const float* v) {
  const uint32_t row = buf + (uint32_t)lane * 64u;
  const int sw = (lane >> 1) & 3;
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    uint32_t w[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      __nv_bfloat162 h2 = __floats2bfloat162_rn(v[8 * j + 2 * i], v[8 * j + 2 * i + 1]);
      w[i] = *reinterpret_cast<uint32_t*>(&h2);
    }
    asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(row + ((uint32_t)(j ^ sw) << 4)),
                 "r"(w[0]), "r"(w[1]), "r"(w[2]), "r"(w[3])
                 : "memory");
  }
}

// One row of a 32-row x 16-column bf16 box (8 values = 16 B chunk j of the
// row's 32 bytes) into a 1 KB half of the warp's buffer, in the 32-byte
// swizzle of its tensor map: chunk j of row r sits at chunk j ^ ((r >> 2) & 1)
// (eight consecutive rows then cover all 32 banks).
__device__ __forceinline__ void stage_box16_chunk(uint32_t buf, int lane, int j, const float* v) {
  uint32_t w[4];
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    __nv_bfloat162 h2 = __floats2bfloat162_rn(v[2 * i], v[2 * i + 1]);
    w[i] = *reinterpret_cast<uint32_t*>(&h2);
  }
  const uint32_t a = buf + (uint32_t)lane * 32u + ((uint32_t)(j ^ ((lane >> 2) & 1)) << 4);
  asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(a), "r"(w[0]), "r"(w[1]),
               "r"(w[2]), "r"(w[3])
               : "memory");
}

// Store the warp's 32 rows x 32 columns through its staging buffer: wait until
// the previous box has left the buffer, stage, hand it to the TMA unit. The
// tensor map clips rows and columns outside the output.
__device__ __forceinline__ void store_box(const CUtensorMap* map, uint32_t buf, int lane,
                                          const float* v, int x, int y) {
  if (lane == 0) bulk_wait_read<0>();
  __syncwarp();
  stage_box_row(buf, lane, v);
  fence_async_shared();
  __syncwarp();
  if (lane == 0) tma_store_2d(map, buf, x, y);
}

// The same 32 x 32 box written by the warp itself: staged as above, then read
// back as eight rows of 64 bytes per instruction (four lanes per row) and
// stored with coalesced 16-byte stores; rows at or past rows_valid and columns
// at or past cols_valid (a multiple of 8) are skipped. No TMA unit is involved
// and the buffer is free again when the function returns.
__device__ __forceinline__ void store_box_rows(uint32_t buf, int lane, const float* v, bf16* dst,
                                               int64_t ld, int64_t rows_valid, int cols_valid) {
  __syncwarp();
  stage_box_row(buf, lane, v);
  __syncwarp();
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const int r = i * 8 + (lane >> 2), ch = lane & 3;
    uint32_t w0, w1, w2, w3;
    asm volatile("ld.shared.v4.b32 {%0, %1, %2, %3}, [%4];"
                 : "=r"(w0), "=r"(w1), "=r"(w2), "=r"(w3)
                 : "r"(buf + (uint32_t)r * 64u + ((uint32_t)(ch ^ ((r >> 1) & 3)) << 4)));
    if (r < rows_valid && ch * 8 < cols_valid)
      *reinterpret_cast<uint4*>(dst + (int64_t)r * ld + ch * 8) = make_uint4(w0, w1, w2, w3);
  }
  __syncwarp();
}

// ---------------------------------------------------------------- tile schedule
struct Tile {
  int grp;
  int m0;       // M-grouped: first row (absolute); K-grouped: first output row
  int m_end;    // row limit for stores
  int n0;       // first output column (SwiGLU fwd: first gate column)
  int k_begin;  // K-grouped: first row of the segment
  int k_end;
  int nk;       // k-blocks
  int m128;     // CTA pair: a segment's last tile of at most 128 rows, computed
                // with M = 128 (64 rows per CTA)
};

// Which accumulator cells an epilogue thread drains. TMEM lane = accumulator
// row, except in an M = 128 pair tile, whose 64 rows x 256 columns per CTA
// sit folded in 128 lanes x 128 columns: lanes 0-63 hold columns 0-127 and
// lanes 64-127 hold columns 128-255 of the same 64 rows (measured).
struct EpiCols {
  int row;      // accumulator row of this thread, relative to the tile's m0
  int cb, ncol; // TMEM columns [cb, cb + ncol) of this warp (plain outputs)
  int dbase;    // output column of TMEM column 0 for this thread's lanes
  int gcol;     // SwiGLU forward: TMEM column of the first gate value,
  int up_off;   //   the matching up value up_off columns further,
  int feat_off; //   its feature index relative to the tile's n0,
  int nchunk;   //   and how many 32-feature chunks this warp takes
};
__device__ __forceinline__ EpiCols epi_cols(int q, int lane, int half, bool pair_glu, bool m128) {
  EpiCols e;
  if (!m128) {
    e.row = q * 32 + lane;
    e.cb = half * (BN / 2);
    e.ncol = BN / 2;
    e.dbase = 0;
    if (pair_glu) {  // CTA pair: B = [64 gate | 64 up] rows per CTA
      e.gcol = half * (BN / 2);
      e.up_off = BN / 4;
    } else {         // single CTA: B = [128 gate | 128 up] rows
      e.gcol = half * (BN / 4);
      e.up_off = BN / 2;
    }
    e.feat_off = half * (BN / 4);
    e.nchunk = 2;
  } else {
    e.row = (q & 1) * 32 + lane;
    e.cb = half * (BN / 4);
    e.ncol = BN / 4;
    e.dbase = q >= 2 ? BN / 2 : 0;
    e.gcol = half * 32;
    e.up_off = BN / 4;
    e.feat_off = (q >= 2 ? BN / 4 : 0) + half * 32;
    e.nchunk = 1;
  }
  return e;
}

template <bool KGROUPED, int EPI>
__device__ __forceinline__ Tile decode_tile(const Shared& sh, const Params& P, int t) {
  Tile ti;
  if (!KGROUPED) {
    int lo = 0, hi = P.G;
    while (hi - lo > 1) {
      const int mid = (lo + hi) >> 1;
      if (sh.prefix[mid] <= t) lo = mid; else hi = mid;
    }
    const int g = lo;
    const int rows = sh.off[g + 1] - sh.off[g];
    const int mt = (rows + BM - 1) / BM;
    const int local = t - sh.prefix[g];
    const int ni = local / mt, mi = local - ni * mt;
    ti.grp = g;
    ti.m0 = sh.off[g] + mi * BM;
    ti.m_end = sh.off[g + 1];
    ti.n0 = ni * (EPI == EPI_SWIGLU_FWD ? BN / 2 : BN);
    ti.k_begin = 0;
    ti.k_end = P.K;
    ti.nk = (P.K + BK - 1) / BK;
    ti.m128 = 0;
  } else {
    const int per = P.MT * P.NT;
    const int gi = t / per;
    const int local = t - gi * per;
    const int g = sh.order[gi];
    const int mi = local / P.NT, ni = local - mi * P.NT;
    ti.grp = g;
    ti.m0 = mi * BM;
    ti.m_end = P.M_out;
    ti.n0 = ni * BN;
    ti.k_begin = sh.off[g];
    ti.k_end = sh.off[g + 1];
    ti.nk = (ti.k_end - ti.k_begin + BK - 1) / BK;
    ti.m128 = 0;
  }
  return ti;
}

// ---------------------------------------------------------------- epilogues
// One thread per accumulator row (TMEM lane): read the row's 256 fp32 columns
// with tcgen05.ld (all lanes of the warp together) and write the outputs.
template <int EPI>
__device__ __forceinline__ bool drain_tile(const Params& P, const Tile& ti, uint32_t t_row,
                                           const EpiCols& ec, const CUtensorMap* tmC,
                                           const CUtensorMap* tmD, uint32_t ebuf,
                                           uint64_t* load_bar, uint32_t& load_phase,
                                           int& abort_flag) {
  // the two warps of a lane quadrant split the accumulator's columns in halves
  const int lane = ec.row & 31;
  if (EPI == EPI_SWIGLU_FWD) {
    const int r = ti.m0 + ec.row;
    const bool rv = r < ti.m_end;
    // whole 32 x 32 boxes through the TMA unit (h: tmC, gate|up: tmD) when the
    // warp's 32 rows are in the segment and the 32 columns inside F (a gate
    // box past F would land on the up columns of the same rows)
    const int y0 = r - lane;
    const bool rows_boxed = P.tma_out && y0 + 32 <= ti.m_end;
#pragma unroll 1
    for (int k = 0; k < ec.nchunk; ++k) {
      float g[32], u[32];
      tmem_ld32(t_row + ec.gcol + 32 * k, g);
      tmem_ld32(t_row + ec.gcol + ec.up_off + 32 * k, u);
      const int f0 = ti.n0 + ec.feat_off + 32 * k;
      const bool boxed = rows_boxed && f0 + 32 <= P.F;
      if (boxed && P.out1) {
        store_box(tmD, ebuf, lane, g, f0, y0);
        store_box(tmD, ebuf, lane, u, P.F + f0, y0);
      } else if (rv && P.out1) {
        // the pre-activation gate|up first: h then overwrites g in place
        bf16* pr = P.out1 + (int64_t)r * 2 * P.F;
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          if (f0 + 8 * j < P.F) {
            store_bf16x8(pr + f0 + 8 * j, g + 8 * j);
            store_bf16x8(pr + P.F + f0 + 8 * j, u + 8 * j);
          }
        }
      }
      if (glu_is_plain(P.act)) {
#pragma unroll
        for (int i = 0; i < 32; ++i) g[i] = silu_f(g[i]) * u[i];
      } else {
#pragma unroll
        for (int i = 0; i < 32; ++i) g[i] = glu_fwd(g[i], u[i], P.act);
      }
      if (boxed) {
        store_box(tmC, ebuf, lane, g, f0, y0);
      } else if (rv) {
#pragma unroll
        for (int j = 0; j < 4; ++j)
          if (f0 + 8 * j < P.F) store_bf16x8(P.out0 + (int64_t)r * P.ld0 + f0 + 8 * j, g + 8 * j);
      }
    }
  } else if (EPI == EPI_STORE) {
    const int r = ti.m0 + ec.row;
    const bool rv = r < ti.m_end;
    // the warp's 32 rows all in the segment: whole boxes through the TMA unit
    const int y0 = r - lane;
    const bool boxed = P.tma_out && y0 + 32 <= ti.m_end;
#pragma unroll 1
    for (int ct = ec.cb; ct < ec.cb + ec.ncol; ct += 32) {
      float v[32];
      tmem_ld32(t_row + ct, v);
      const int c = ec.dbase + ct;  // accumulator column
      if (boxed) {
        if (ti.n0 + c < P.N_out) store_box(tmC, ebuf, lane, v, ti.n0 + c, y0);
      } else if (rv) {
#pragma unroll
        for (int j = 0; j < 4; ++j)
          if (ti.n0 + c + 8 * j < P.N_out)
            store_bf16x8(P.out0 + (int64_t)r * P.ld0 + ti.n0 + c + 8 * j, v + 8 * j);
      }
    }
  } else if (EPI == EPI_SWIGLU_BWD) {
    // The warp's 32 rows inside the segment and the columns inside F: gate/up
    // come in and d_pre goes out through the warp's buffer, 16 columns at a
    // time, as 32 x 16 boxes in the 32-byte swizzle (tmD: gate|up, tmC:
    // d_pre; each a 3-D map whose one copy moves the box of both halves, the
    // gate or dg box then the up or du box, 1 KB apart: half the TMA copies
    // of two 2-D boxes, measured 1% faster); each thread reads its row's
    // chunks and writes dg/du in place. Elsewhere each thread loads and
    // stores its row directly.
    const int r = ti.m0 + ec.row;
    const bool rv = r < ti.m_end;
    const int y0 = r - lane;
    const bool rows_boxed = P.tma_out && y0 + 32 <= ti.m_end;
    const bf16* pr = P.aux_in + (int64_t)(rv ? r : ti.m0) * 2 * P.F;
    bf16* dp = P.out0 + (int64_t)r * 2 * P.F;
    auto deriv8 = [&](const float* gv, const float* uv, const float* d, float* dg, float* du) {
      if (glu_is_plain(P.act)) {
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          const float sg = 1.f / (1.f + __expf(-gv[i]));
          dg[i] = d[i] * uv[i] * sg * (1.f + gv[i] * (1.f - sg));
          du[i] = d[i] * gv[i] * sg;
        }
      } else {
#pragma unroll
        for (int i = 0; i < 8; ++i) glu_bwd(gv[i], uv[i], d[i], P.act, dg[i], du[i]);
      }
    };
#pragma unroll 1
    for (int ct = ec.cb; ct < ec.cb + ec.ncol; ct += 32) {
      float dh[32];
      tmem_ld32(t_row + ct, dh);
      const int fc = ti.n0 + ec.dbase + ct;
      if (rows_boxed && fc + 32 <= P.F) {
#pragma unroll
        for (int s2 = 0; s2 < 2; ++s2) {
          const int x = fc + 16 * s2;
          if (lane == 0) {
            bulk_wait_read<0>();  // the previous boxes have left the buffer
            mbar_expect_tx(load_bar, 2048);
            tma_load_3d_s(ebuf, tmD, su32(load_bar), x, y0, 0);
          }
          if (!mbar_wait(load_bar, load_phase, abort_flag, P, 16)) return false;
          load_phase ^= 1;
#pragma unroll
          for (int jj = 0; jj < 2; ++jj) {
            const uint32_t off = (uint32_t)lane * 32u + ((uint32_t)(jj ^ ((lane >> 2) & 1)) << 4);
            uint4 gq, uq;
            asm volatile("ld.shared.v4.b32 {%0, %1, %2, %3}, [%4];"
                         : "=r"(gq.x), "=r"(gq.y), "=r"(gq.z), "=r"(gq.w)
                         : "r"(ebuf + off));
            asm volatile("ld.shared.v4.b32 {%0, %1, %2, %3}, [%4];"
                         : "=r"(uq.x), "=r"(uq.y), "=r"(uq.z), "=r"(uq.w)
                         : "r"(ebuf + 1024 + off));
            float gv[8], uv[8], dg[8], du[8];
            const __nv_bfloat162* g2 = reinterpret_cast<const __nv_bfloat162*>(&gq);
            const __nv_bfloat162* u2 = reinterpret_cast<const __nv_bfloat162*>(&uq);
#pragma unroll
            for (int i = 0; i < 4; ++i) {
              const float2 a = __bfloat1622float2(g2[i]);
              const float2 b2 = __bfloat1622float2(u2[i]);
              gv[2 * i] = a.x; gv[2 * i + 1] = a.y;
              uv[2 * i] = b2.x; uv[2 * i + 1] = b2.y;
            }
            deriv8(gv, uv, dh + 16 * s2 + 8 * jj, dg, du);
            stage_box16_chunk(ebuf, lane, jj, dg);
            stage_box16_chunk(ebuf + 1024, lane, jj, du);
          }
          fence_async_shared();
          __syncwarp();
          if (lane == 0) tma_store_3d(tmC, ebuf, x, y0, 0);
        }
      } else if (rv) {
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          const int f = fc + 8 * j;
          if (f < P.F) {
            float gv[8], uv[8], dg[8], du[8];
            load_bf16x8(pr + f, gv);
            load_bf16x8(pr + P.F + f, uv);
            deriv8(gv, uv, dh + 8 * j, dg, du);
            store_bf16x8(dp + f, dg);
            store_bf16x8(dp + P.F + f, du);
          }
        }
      }
    }
  } else {  // EPI_WGRAD
    // The weight gradients' boxes leave through the warp's own coalesced
    // stores (store_box_rows), not TMA stores: the TMA unit of these kernels
    // also issues four operand loads per stage, and taking the outputs off it
    // measured 4-5% faster weight-gradient kernels on Mixtral-style shapes.
    const int m = ti.m0 + ec.row;
    const bool rv = m < P.M_out;
    bf16* dst_row = P.out0 + (int64_t)ti.grp * P.M_out * P.N_out + (int64_t)m * P.N_out;
#pragma unroll 1
    for (int c = ec.cb; c < ec.cb + ec.ncol; c += 32) {
      float v[32];
      tmem_ld32(t_row + c, v);
      if (P.tma_out) {  // rows 16-byte aligned: staged boxes
        if (ti.n0 + c < P.N_out && m - lane < P.M_out)
          store_box_rows(ebuf, lane, v, dst_row - (int64_t)lane * P.N_out + ti.n0 + c, P.N_out,
                         P.M_out - (m - lane), P.N_out - (ti.n0 + c));
      } else if (rv) {
#pragma unroll
        for (int j = 0; j < 4; ++j)
          if (ti.n0 + c + 8 * j < P.N_out) store_bf16x8(dst_row + ti.n0 + c + 8 * j, v + 8 * j);
      }
    }
  }
  return true;
}

// An empty expert's weight-gradient tile: zeros, without touching TMEM.
__device__ __forceinline__ void zero_wgrad_tile(const Params& P, const Tile& ti, int row_in_tile,
                                                int half, const CUtensorMap* tmC, uint32_t ebuf) {
  const int m = ti.m0 + row_in_tile;
  if (P.tma_out) {
    const int lane = row_in_tile & 31;
    float z[32];
#pragma unroll
    for (int i = 0; i < 32; ++i) z[i] = 0.f;
    bf16* dst0 = P.out0 + (int64_t)ti.grp * P.M_out * P.N_out + (int64_t)(m - lane) * P.N_out;
    for (int c = half * (BN / 2); c < (half + 1) * (BN / 2); c += 32)
      if (ti.n0 + c < P.N_out && m - lane < P.M_out)
        store_box_rows(ebuf, lane, z, dst0 + ti.n0 + c, P.N_out, P.M_out - (m - lane),
                       P.N_out - (ti.n0 + c));
  } else if (m < P.M_out) {
    bf16* dst_row = P.out0 + (int64_t)ti.grp * P.M_out * P.N_out + (int64_t)m * P.N_out;
    const float z[8] = {0, 0, 0, 0, 0, 0, 0, 0};
    for (int c = half * (BN / 2); c < (half + 1) * (BN / 2); c += 8)
      if (ti.n0 + c < P.N_out) store_bf16x8(dst_row + ti.n0 + c, z);
  }
}

// ---------------------------------------------------------------- the kernel
// GATHER (M-grouped, K-major A): the A tile is not loaded by TMA from a
// permuted copy but gathered row by row from a_rows through a_src (the
// dispatch's src_tok), by the producer warp's 32 lanes with 16-byte cp.async
// copies written in the 128-byte swizzle the MMA descriptors expect. A lane
// keeps GATHER_LAG stages of its copies in flight; once a stage's copies have
// landed it fences them towards the async proxy (which the MMA reads through)
// and arrives on the stage's `full` barrier, which also waits for the B tile's
// TMA bytes.
constexpr int GATHER_LAG = STAGES - 1;

template <bool A_MN, bool B_MN, int EPI, bool GATHER = false>
__global__ void __launch_bounds__(NUM_THREADS, 1)
tc_grouped_gemm(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                const __grid_constant__ CUtensorMap tmC, const __grid_constant__ CUtensorMap tmD,
                const Params P) {
  static_assert(!GATHER || (!A_MN && EPI != EPI_WGRAD), "gather: M-grouped, K-major A");
  constexpr bool KGROUPED = (EPI == EPI_WGRAD);
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  // 1024-byte alignment for the swizzled stages
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  uint8_t* stage_base = smem;
  uint8_t* epi_buf = smem + STAGES * STAGE_BYTES;  // 1024-byte aligned
  Shared& sh = *reinterpret_cast<Shared*>(smem + STAGES * STAGE_BYTES + EPI_BUF_BYTES);

  const int tid = threadIdx.x;
  const int warp = tid >> 5;
  const int lane = tid & 31;
  const int tile0 = (int)blockIdx.x;
  const int tstep = (int)gridDim.x;

  // ---- set-up: barriers, TMEM, then (once the kernel before has finished:
  // this kernel is a dependent launch) segment offsets and the tile prefix
  if (tid == 0) {
    sh.abort = 0;
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(&sh.full[s], GATHER ? 33 : 1);  // gather: + one arrival per producer lane
      mbar_init(&sh.empty[s], 1);
    }
    for (int a = 0; a < 2; ++a) {
      mbar_init(&sh.tmem_full[a], 1);
      mbar_init(&sh.tmem_empty[a], NUM_EPI_WARPS);  // one arrival per epilogue warp
    }
    for (int w = 0; w < NUM_EPI_WARPS; ++w) mbar_init(&sh.epi_load[w], 1);
    fence_barrier_init();
  }
  if (warp == 1) {
    tmem_alloc(&sh.tmem_base, TMEM_COLS);
    tmem_relinquish();
  }
  if (warp == 0 && lane == 0) {
    prefetch_tmap(&tmA);
    prefetch_tmap(&tmB);
  }
  pdl_wait();
  for (int g = tid; g <= P.G; g += NUM_THREADS) {
    int v = P.offsets ? P.offsets[g] : (g == 0 ? 0 : P.n_rows);
    sh.off[g] = v;
  }
  __syncthreads();
  if (tid == 0) {
    // validate: monotone, within [0, n_rows]; a bad segment becomes empty
    int prev = 0;
    bool bad = false;
    for (int g = 0; g <= P.G; ++g) {
      int v = sh.off[g];
      if (v < prev || v > P.n_rows || (g == 0 && v != 0)) {
        bad = true;
        v = prev;
      }
      sh.off[g] = v;
      prev = v;
    }
    if (bad) record_error(P.status, MOE_ERR_DEVICE_INDEX, -1);
    if (!KGROUPED) {
      int acc = 0;
      for (int g = 0; g < P.G; ++g) {
        sh.prefix[g] = acc;
        acc += ((sh.off[g + 1] - sh.off[g] + BM - 1) / BM) * P.NT;
      }
      sh.prefix[P.G] = acc;
      sh.total_tiles = acc;
    } else {
      sh.total_tiles = P.G * P.MT * P.NT;
    }
  }
  if (KGROUPED) {
    __syncthreads();
    // longest segment first; ties by group index
    for (int g = tid; g < P.G; g += NUM_THREADS) {
      const int ng = sh.off[g + 1] - sh.off[g];
      int rank = 0;
      for (int h = 0; h < P.G; ++h) {
        const int nh = sh.off[h + 1] - sh.off[h];
        rank += (nh > ng) || (nh == ng && h < g);
      }
      sh.order[rank] = g;
    }
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();

  const int total = sh.total_tiles;
  const uint32_t tmem_base = sh.tmem_base;

  if (warp == 0 && GATHER) {
    // ================= producer: gathered A rows (cp.async) + B by TMA =================
    const int nchunk = P.K >> 3;  // 16-byte chunks per A row
    int stage = 0;
    uint32_t phase = 0;
    int pend_stage[GATHER_LAG + 1];
    int npend = 0;
    bool ok = true;
    auto release_oldest = [&]() {  // the oldest pending stage's copies have landed
      fence_async_shared();
      mbar_arrive(&sh.full[pend_stage[0]]);
#pragma unroll
      for (int i = 0; i < GATHER_LAG; ++i) pend_stage[i] = pend_stage[i + 1];
      --npend;
    };
    for (int t = tile0; t < total && ok; t += tstep) {
      const Tile ti = decode_tile<KGROUPED, EPI>(sh, P, t);
      // this lane's four rows of the tile: r = lane + 32 i
      const bf16* src[4];
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const int r = ti.m0 + lane + 32 * i;
        int s_row = -1;
        if (r < P.n_rows) s_row = P.a_src[r];
        src[i] = (s_row >= 0 && s_row < P.a_src_rows) ? P.a_rows + (int64_t)s_row * P.K : nullptr;
      }
      for (int kb = 0; kb < ti.nk; ++kb) {
        if (!mbar_wait(&sh.empty[stage], phase ^ 1, sh.abort, P, 5)) { ok = false; break; }
        uint8_t* a_dst = stage_base + stage * STAGE_BYTES;
        uint8_t* b_dst = a_dst + A_STAGE_BYTES;
        if (lane == 0) {
          uint64_t* bar = &sh.full[stage];
          mbar_expect_tx(bar, B_STAGE_BYTES);
          const int k0 = kb * BK;
          if (EPI == EPI_SWIGLU_FWD) {
            const int r0 = ti.grp * 2 * P.F;
            for (int h = 0; h < 2; ++h)
              tma_load_2d(b_dst + 16384 * h, &tmB, bar, k0, r0 + h * P.F + ti.n0);
          } else {
            tma_load_2d(b_dst, &tmB, bar, k0, ti.grp * P.b_group_rows + ti.n0);
          }
        }
        const uint32_t a_s = su32(a_dst);
        const int c0 = kb * (BK / 8);  // first 16-byte chunk of this K block
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          const int r = lane + 32 * i;
#pragma unroll
          for (int c = 0; c < 8; ++c) {
            const bool in = src[i] != nullptr && c0 + c < nchunk;
            const void* g = in ? static_cast<const void*>(src[i] + 8 * (c0 + c))
                               : static_cast<const void*>(P.a_rows);
            cp_async16_zfill(a_s + r * 128 + ((c ^ (r & 7)) << 4), g, in ? 16u : 0u);
          }
        }
        cp_async_commit();
        pend_stage[npend++] = stage;
        if (npend > GATHER_LAG) {
          cp_async_wait_group<GATHER_LAG>();
          release_oldest();
        }
        if (++stage == STAGES) { stage = 0; phase ^= 1; }
      }
    }
    cp_async_wait_all();
    while (npend > 0) release_oldest();
    if (!ok) {
      const uint64_t t0 = global_timer_ns();
      while (global_timer_ns() - t0 < 2000000ull) { }
    }
  } else if (warp == 0) {
    // ================= TMA producer =================
    // Loads run up to STAGES k-blocks ahead of the MMAs. (An L2 prefetch of
    // later k-blocks by every CTA was measured to slow the kernel down: the
    // CTAs sharing a weight tile all prefetch it.)
    if (lane == 0) {
      // the A and B boxes of k-block kb of tile ti
      auto kblock = [&](const Tile& ti, int kb, uint8_t* a_dst, uint8_t* b_dst, uint64_t* bar) {
        const int k0 = kb * BK;
        if (!A_MN) {
          tma_load_2d(a_dst, &tmA, bar, k0, ti.m0);
        } else {
          for (int h = 0; h < 2; ++h)
            tma_load_2d(a_dst + 8192 * h, &tmA, bar, ti.m0 + 64 * h, ti.k_begin + k0);
        }
        if (!B_MN) {
          if (EPI == EPI_SWIGLU_FWD) {
            const int r0 = ti.grp * 2 * P.F;
            for (int h = 0; h < 2; ++h)
              tma_load_2d(b_dst + 16384 * h, &tmB, bar, k0, r0 + h * P.F + ti.n0);
          } else {
            tma_load_2d(b_dst, &tmB, bar, k0, ti.grp * P.b_group_rows + ti.n0);
          }
        } else {
          const int y = KGROUPED ? ti.k_begin + k0 : ti.grp * P.b_group_rows + k0;
          for (int j = 0; j < 4; ++j) tma_load_2d(b_dst + j * 8192, &tmB, bar, ti.n0 + 64 * j, y);
        }
      };
      int stage = 0;
      uint32_t phase = 0;
      bool ok = true;
      for (int t = tile0; t < total && ok; t += tstep) {
        const Tile ti = decode_tile<KGROUPED, EPI>(sh, P, t);
        for (int kb = 0; kb < ti.nk; ++kb) {
          if (!mbar_wait(&sh.empty[stage], phase ^ 1, sh.abort, P, 1)) { ok = false; break; }
          uint8_t* a_dst = stage_base + stage * STAGE_BYTES;
          uint64_t* bar = &sh.full[stage];
          mbar_expect_tx(bar, STAGE_BYTES);
          kblock(ti, kb, a_dst, a_dst + A_STAGE_BYTES, bar);
          if (++stage == STAGES) { stage = 0; phase ^= 1; }
        }
      }
      if (!ok) {
        // let the copies already in flight land before the CTA exits
        const uint64_t t0 = global_timer_ns();
        while (global_timer_ns() - t0 < 2000000ull) { }
      }
    }
  } else if (warp == 1) {
    // ================= MMA issuer (whole warp walks; lane 0 issues; warp 10 waits) =================
    constexpr uint32_t IDESC = make_idesc(A_MN, B_MN);
    int stage = 0;
    int acc = 0;
    for (int t = tile0; t < total; t += tstep) {
      const Tile ti = decode_tile<KGROUPED, EPI>(sh, P, t);
      if (ti.nk == 0) continue;  // empty segment: the epilogue writes zeros itself
      const uint32_t d_tmem = tmem_base + acc * BN;
      for (int kb = 0; kb < ti.nk; ++kb) {
        // the relay warp has seen this stage's tiles land (and, at kb == 0,
        // this accumulator drained by the epilogue)
        warp_pair_sync(RELAY_BAR);
        tc_fence_after();
        uint8_t* a_s = stage_base + stage * STAGE_BYTES;
        uint8_t* b_s = a_s + A_STAGE_BYTES;
        int nkk = BK / 16;  // K16 steps of this stage that hold rows of the segment
        if (KGROUPED && kb == ti.nk - 1) {
          // rows past the segment end belong to the next expert: the K16 steps
          // wholly past it are not issued, and the rest of the last partial one
          // is zeroed in A
          const int valid = ti.k_end - (ti.k_begin + kb * BK);
          if (valid < BK) {
            nkk = (valid + 15) >> 4;
            const int n16 = (nkk * 16 - valid) * 8;
            if (n16 > 0) {
              for (int half = 0; half < 2; ++half) {
                uint4* z = reinterpret_cast<uint4*>(a_s + half * 8192 + valid * 128);
                for (int i = lane; i < n16; i += 32) z[i] = make_uint4(0, 0, 0, 0);
              }
              fence_async_shared();
            }
            __syncwarp();
          }
        }
        if (lane == 0) {
          const uint32_t a_addr = su32(a_s), b_addr = su32(b_s);
#pragma unroll
          for (int kk = 0; kk < BK / 16; ++kk) {
            if (kk >= nkk) break;
            uint64_t ad, bd;
            if (!A_MN) ad = sw128_desc(a_addr + kk * 32, 16, 1024);
            else ad = sw128_desc(a_addr + kk * 2048, 8192, 1024);
            if (!B_MN) bd = sw128_desc(b_addr + kk * 32, 16, 1024);
            else bd = sw128_desc(b_addr + kk * 2048, 8192, 1024);
            mma_bf16(d_tmem, ad, bd, IDESC, (kb | kk) != 0 ? 1u : 0u);
          }
          mma_commit(&sh.empty[stage]);
        }
        __syncwarp();
        if (++stage == STAGES) stage = 0;
      }
      if (lane == 0) mma_commit(&sh.tmem_full[acc]);
      __syncwarp();
      acc ^= 1;
    }
  } else if (warp == RELAY_WARP) {
    relay_waits(sh, P, tile0, tstep, total, [&](int t) { return decode_tile<KGROUPED, EPI>(sh, P, t); },
                STAGES, 2, 2);
  } else {
    // ================= epilogue: warps 2..9 =================
    const int q = warp & 3;  // TMEM lanes 32q .. 32q+31
    const int half = (warp - 2) >> 2;
    const int row_in_tile = q * 32 + lane;
    const uint32_t ebuf = su32(epi_buf) + (uint32_t)(warp - 2) * EPI_BOX_BYTES;
    uint32_t epi_phase = 0;  // parity of this warp's epi_load barrier
    int acc = 0;
    uint32_t acc_phase = 0;
    for (int t = tile0; t < total; t += tstep) {
      const Tile ti = decode_tile<KGROUPED, EPI>(sh, P, t);
      if (EPI == EPI_WGRAD && ti.nk == 0) {
        zero_wgrad_tile(P, ti, row_in_tile, half, &tmC, ebuf);
        continue;
      }
      if (!mbar_wait(&sh.tmem_full[acc], acc_phase, sh.abort, P, 4)) break;
      tc_fence_after();
      const uint32_t t_row = tmem_base + ((uint32_t)(q * 32) << 16) + acc * BN;

      if (!drain_tile<EPI>(P, ti, t_row, epi_cols(q, lane, half, false, false), &tmC, &tmD, ebuf,
                           &sh.epi_load[warp - 2], epi_phase, sh.abort))
        break;
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&sh.tmem_empty[acc]);
      acc ^= 1;
      if (acc == 0) acc_phase ^= 1;
    }
    if (lane == 0) bulk_wait_all();  // this warp's TMA stores have landed
  }

  pdl_launch_dependents();  // this CTA's work is done
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem_base, TMEM_COLS);
  }
}

// ---------------------------------------------------------------- CTA-pair kernel
// The M-grouped contractions on a pair of CTAs (a 2-CTA cluster on two SMs):
// one tcgen05.mma.cta_group::2 instruction computes a 256 x 256 tile whose
// rows 0..127 come from (and accumulate in) the even CTA and rows 128..255 in
// the odd one; each CTA stages only its own 128 rows of A and its own half
// (128 columns) of B. Per SM and per K step that is 32 KB of shared-memory
// traffic each way instead of 48 KB in and 48 KB read by the single-CTA
// kernel, and 6 pipeline stages fit instead of 4.
// Protocol: both CTAs' TMA loads complete on the even CTA's `full` barrier;
// the even CTA issues the MMAs and its commits arrive on both CTAs' `empty`
// and `tmem_full` barriers; every epilogue warp of both CTAs arrives on the
// even CTA's `tmem_empty`.
constexpr int STAGES2 = 6;
constexpr int A2_BYTES = BM * BK * 2;              // 16 KB: this CTA's 128 rows
constexpr int B2_BYTES = (BN / 2) * BK * 2;        // 16 KB: this CTA's half of N
constexpr int STAGE2_BYTES = A2_BYTES + B2_BYTES;  // 32 KB
constexpr int PAIR_ACC = 2;                        // accumulators per CTA (x 256 columns)

struct __align__(8) Shared2 {
  uint64_t full[STAGES2];
  uint64_t empty[STAGES2];
  uint64_t epi_load[NUM_EPI_WARPS];  // TMA loads into an epilogue warp's buffer
  uint64_t tmem_full[PAIR_ACC];
  uint64_t tmem_empty[PAIR_ACC];
  uint32_t tmem_base;
  int abort;
  int total_tiles;
  int off[MAXG + 1];
  int prefix[MAXG + 1];
  int order[MAXG];
};

__device__ __forceinline__ void mbar_arrive_cluster(uint32_t cluster_addr) {
  asm volatile("mbarrier.arrive.release.cluster.shared::cluster.b64 _, [%0];" ::"r"(cluster_addr)
               : "memory");
}
// TMA into this CTA's shared memory, completing on a barrier of either CTA of the pair
__device__ __forceinline__ void tma_load_2d_pair(void* dst, const CUtensorMap* map,
                                                 uint32_t bar_cluster_addr, int x, int y) {
  asm volatile(
      "cp.async.bulk.tensor.2d.cta_group::2.shared::cluster.global.mbarrier::complete_tx::bytes "
      "[%0], [%1, {%2, %3}], [%4];" ::"r"(su32(dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(bar_cluster_addr)
      : "memory");
}
__device__ __forceinline__ void tmem_alloc_pair(uint32_t* dst, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::2.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(su32(dst)),
               "r"(ncols)
               : "memory");
}
__device__ __forceinline__ void tmem_relinquish_pair() {
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::2.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc_pair(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::2.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols)
               : "memory");
}
__device__ __forceinline__ void mma_bf16_pair(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc,
                                              uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::2.kind::f16 [%0], %1, %2, %3, p;\n\t}\n" ::"r"(d_tmem),
      "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
      : "memory");
}
// arrive on the barrier at this offset in every CTA of `mask`
__device__ __forceinline__ void mma_commit_pair(uint64_t* bar, uint16_t mask) {
  asm volatile(
      "tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64 "
      "[%0], %1;" ::"r"(su32(bar)),
      "h"(mask)
      : "memory");
}

__host__ __device__ constexpr uint32_t make_idesc_pair(bool a_mn, bool b_mn) {
  return (1u << 4) | (1u << 7) | (1u << 10) | ((a_mn ? 1u : 0u) << 15) |
         ((b_mn ? 1u : 0u) << 16) | ((uint32_t)(BN >> 3) << 17) | ((uint32_t)((2 * BM) >> 4) << 24);
}

template <bool KGROUPED, int EPI>
__device__ __forceinline__ Tile decode_pair_tile(const Shared2& sh, const Params& P, int t,
                                                 uint32_t rank) {
  Tile ti;
  if (!KGROUPED) {
    int lo = 0, hi = P.G;
    while (hi - lo > 1) {
      const int mid = (lo + hi) >> 1;
      if (sh.prefix[mid] <= t) lo = mid; else hi = mid;
    }
    const int g = lo;
    const int rows = sh.off[g + 1] - sh.off[g];
    const int mp = (rows + 2 * BM - 1) / (2 * BM);
    const int local = t - sh.prefix[g];
    const int ni = local / mp, mi = local - ni * mp;
    // a last tile of at most 128 rows runs as M = 128: 64 rows per CTA
    const bool m128 = P.m128_tails && mi == mp - 1 && rows - mi * 2 * BM <= BM;
    ti.grp = g;
    ti.m0 = sh.off[g] + mi * 2 * BM + (int)rank * (m128 ? BM / 2 : BM);
    ti.m_end = sh.off[g + 1];
    ti.n0 = ni * (EPI == EPI_SWIGLU_FWD ? BN / 2 : BN);
    ti.k_begin = 0;
    ti.k_end = P.K;
    ti.nk = (P.K + BK - 1) / BK;
    ti.m128 = m128 ? 1 : 0;
  } else {
    // P.MT counts 256-row pair tiles along M
    const int per = P.MT * P.NT;
    const int gi = t / per;
    const int local = t - gi * per;
    const int g = sh.order[gi];
    const int mi = local / P.NT, ni = local - mi * P.NT;
    ti.grp = g;
    ti.m0 = mi * 2 * BM + (int)rank * BM;
    ti.m_end = P.M_out;
    ti.n0 = ni * BN;
    ti.k_begin = sh.off[g];
    ti.k_end = sh.off[g + 1];
    ti.nk = (ti.k_end - ti.k_begin + BK - 1) / BK;
    ti.m128 = 0;
  }
  return ti;
}

template <bool A_MN, bool B_MN, int EPI>
__global__ void __launch_bounds__(NUM_THREADS, 1)
tc_grouped_gemm_pair(const __grid_constant__ CUtensorMap tmA,
                     const __grid_constant__ CUtensorMap tmB,
                     const __grid_constant__ CUtensorMap tmC,
                     const __grid_constant__ CUtensorMap tmD,
                     const __grid_constant__ CUtensorMap tmA64, const Params P) {
  constexpr bool KGROUPED = (EPI == EPI_WGRAD);
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  uint8_t* stage_base = smem;
  uint8_t* epi_buf = smem + STAGES2 * STAGE2_BYTES;  // 1024-byte aligned
  Shared2& sh = *reinterpret_cast<Shared2*>(smem + STAGES2 * STAGE2_BYTES + EPI_BUF_BYTES);

  const int tid = threadIdx.x;
  const int warp = tid >> 5;
  const int lane = tid & 31;
  const uint32_t rank = cluster_ctarank();
  const bool leader = (rank == 0);
  const int cluster_id = blockIdx.x >> 1;
  const int n_clusters = gridDim.x >> 1;

  if (tid == 0) {
    sh.abort = 0;
    for (int s2 = 0; s2 < STAGES2; ++s2) {
      mbar_init(&sh.full[s2], 1);
      mbar_init(&sh.empty[s2], 1);
    }
    for (int a = 0; a < PAIR_ACC; ++a) {
      mbar_init(&sh.tmem_full[a], 1);
      mbar_init(&sh.tmem_empty[a], 2 * NUM_EPI_WARPS);
    }
    for (int w = 0; w < NUM_EPI_WARPS; ++w) mbar_init(&sh.epi_load[w], 1);
    fence_barrier_init();
  }
  if (warp == 1) {
    tmem_alloc_pair(&sh.tmem_base, PAIR_ACC * BN);
    tmem_relinquish_pair();
  }
  if (warp == 0 && lane == 0) {
    prefetch_tmap(&tmA);
    prefetch_tmap(&tmB);
  }
  pdl_wait();  // a dependent launch: the offsets come from the kernel before
  for (int g = tid; g <= P.G; g += NUM_THREADS)
    sh.off[g] = P.offsets ? P.offsets[g] : (g == 0 ? 0 : P.n_rows);
  __syncthreads();
  if (tid == 0) {
    int prev = 0;
    bool bad = false;
    for (int g = 0; g <= P.G; ++g) {
      int v = sh.off[g];
      if (v < prev || v > P.n_rows || (g == 0 && v != 0)) {
        bad = true;
        v = prev;
      }
      sh.off[g] = v;
      prev = v;
    }
    if (bad && leader) record_error(P.status, MOE_ERR_DEVICE_INDEX, -1);
    if (!KGROUPED) {
      int acc = 0;
      for (int g = 0; g < P.G; ++g) {
        sh.prefix[g] = acc;
        acc += ((sh.off[g + 1] - sh.off[g] + 2 * BM - 1) / (2 * BM)) * P.NT;
      }
      sh.prefix[P.G] = acc;
      sh.total_tiles = acc;
    } else {
      sh.total_tiles = P.G * P.MT * P.NT;
    }
  }
  if (KGROUPED) {
    __syncthreads();
    for (int g = tid; g < P.G; g += NUM_THREADS) {  // longest segment first
      const int ng = sh.off[g + 1] - sh.off[g];
      int r = 0;
      for (int h = 0; h < P.G; ++h) {
        const int nh = sh.off[h + 1] - sh.off[h];
        r += (nh > ng) || (nh == ng && h < g);
      }
      sh.order[r] = g;
    }
  }
  tc_fence_before();
  __syncthreads();
  cluster_barrier();  // both CTAs' barriers and TMEM exist before any remote access
  tc_fence_after();

  // both CTAs must hold their accumulators at the same TMEM address
  const uint32_t tmem_base = sh.tmem_base;
  const uint32_t peer_base = ld_shared_cluster_u32(mapa_shared(su32(&sh.tmem_base), rank ^ 1u));
  const bool usable = (peer_base == tmem_base);
  if (!usable && tid == 0 && leader) record_error(P.status, MOE_ERR_CUDA, 2000);
  const int total = usable ? sh.total_tiles : 0;
  bool aborted = false;

  if (warp == 0) {
    // ================= TMA producer (both CTAs) =================
    if (lane == 0) {
      int stage = 0;
      uint32_t phase = 0;
      for (int t = cluster_id; t < total && !aborted; t += n_clusters) {
        const Tile ti = decode_pair_tile<KGROUPED, EPI>(sh, P, t, rank);
        for (int kb = 0; kb < ti.nk; ++kb) {
          if (!mbar_wait(&sh.empty[stage], phase ^ 1, sh.abort, P, 11)) { aborted = true; break; }
          uint8_t* a_dst = stage_base + stage * STAGE2_BYTES;
          uint8_t* b_dst = a_dst + A2_BYTES;
          const uint32_t bar = mapa_shared(su32(&sh.full[stage]), 0);  // the even CTA's
          // an M = 128 tile loads only its 64 A rows per CTA (tmA64: 64-row boxes)
          if (leader) mbar_expect_tx(&sh.full[stage], 2 * (ti.m128 ? STAGE2_BYTES - A2_BYTES / 2
                                                                   : STAGE2_BYTES));
          const int k0 = kb * BK;
          const CUtensorMap* amap = &tmA;
          if (KGROUPED && P.tail_maps != nullptr && kb == ti.nk - 1 &&
              ti.k_end - ti.k_begin - k0 < BK && ti.k_end < P.n_rows) {
            // the expert's last block through its own map: the next expert's
            // rows arrive as zeros (past the last row the common map does that)
            amap = P.tail_maps + ti.grp;
            tensormap_acquire(amap);
          }
          if (!A_MN) {
            if (ti.m128) tma_load_2d_pair(a_dst, &tmA64, bar, k0, ti.m0);
            else tma_load_2d_pair(a_dst, amap, bar, k0, ti.m0);
          } else {
            tma_load_2d_pair(a_dst, amap, bar, ti.m0, ti.k_begin + k0);
            tma_load_2d_pair(a_dst + 8192, amap, bar, ti.m0 + 64, ti.k_begin + k0);
          }
          if (!B_MN) {
            if (EPI == EPI_SWIGLU_FWD) {
              // this CTA's 64 features: their gate rows, then their up rows
              const int yg = ti.grp * 2 * P.F + ti.n0 + (int)rank * (BN / 4);
              tma_load_2d_pair(b_dst, &tmB, bar, k0, yg);
              tma_load_2d_pair(b_dst + 8192, &tmB, bar, k0, yg + P.F);
            } else {
              tma_load_2d_pair(b_dst, &tmB, bar, k0,
                               ti.grp * P.b_group_rows + ti.n0 + (int)rank * (BN / 2));
            }
          } else {
            const int y = KGROUPED ? ti.k_begin + k0 : ti.grp * P.b_group_rows + k0;
            const int x0 = ti.n0 + (int)rank * (BN / 2);
            tma_load_2d_pair(b_dst, &tmB, bar, x0, y);
            tma_load_2d_pair(b_dst + 8192, &tmB, bar, x0 + 64, y);
          }
          if (++stage == STAGES2) { stage = 0; phase ^= 1; }
        }
      }
    }
  } else if (warp == 1) {
    // ================= MMA issuer (the even CTA) =================
    if (leader) {
      constexpr uint32_t IDESC = make_idesc_pair(A_MN, B_MN);  // M = 256
      constexpr uint32_t IDESC128 = (IDESC & ~(0x1Fu << 24)) | ((uint32_t)(BM >> 4) << 24);
      int stage = 0;
      int acc = 0;
      for (int t = cluster_id; t < total; t += n_clusters) {
        const Tile ti = decode_pair_tile<KGROUPED, EPI>(sh, P, t, rank);
        if (ti.nk == 0) continue;  // empty segment: the epilogues write zeros themselves
        const uint32_t d_tmem = tmem_base + acc * BN;
        const uint32_t idesc = ti.m128 ? IDESC128 : IDESC;
        for (int kb = 0; kb < ti.nk; ++kb) {
          // the relay warp has seen both CTAs' tiles of this stage land (and,
          // at kb == 0, this accumulator drained by both CTAs' epilogues)
          warp_pair_sync(RELAY_BAR);
          tc_fence_after();
          uint8_t* a_s = stage_base + stage * STAGE2_BYTES;
          int nkk = BK / 16;  // K16 steps of this stage that hold rows of the segment
          if (KGROUPED && kb == ti.nk - 1) {
            // K rows past the segment end belong to the next expert: the K16
            // steps wholly past it are not issued, and the rest of the last
            // partial one arrives as zeros through the expert's own A map, or
            // without the maps is zeroed here in both CTAs' A (this CTA's
            // directly, the peer's through DSMEM)
            const int valid = ti.k_end - (ti.k_begin + kb * BK);
            if (valid < BK) {
              nkk = (valid + 15) >> 4;
              const int n16 = (nkk * 16 - valid) * 8;
              if (n16 > 0 && P.tail_maps == nullptr) {
                for (int half = 0; half < 2; ++half) {
                  uint4* z = reinterpret_cast<uint4*>(a_s + half * 8192 + valid * 128);
                  const uint32_t zp = mapa_shared(su32(z), 1u);
                  for (int i = lane; i < n16; i += 32) {
                    z[i] = make_uint4(0, 0, 0, 0);
                    st_shared_cluster_zero16(zp + 16u * i);
                  }
                }
                fence_async_shared_cluster();
              }
              __syncwarp();
            }
          }
          if (lane == 0) {
            const uint32_t a_addr = su32(a_s);
            const uint32_t b_addr = a_addr + A2_BYTES;
            auto issue = [&](int kk) {
              const uint64_t ad = A_MN ? sw128_desc(a_addr + kk * 2048, 8192, 1024)
                                       : sw128_desc(a_addr + kk * 32, 16, 1024);
              const uint64_t bd = B_MN ? sw128_desc(b_addr + kk * 2048, 8192, 1024)
                                       : sw128_desc(b_addr + kk * 32, 16, 1024);
              mma_bf16_pair(d_tmem, ad, bd, idesc, (kb | kk) != 0 ? 1u : 0u);
            };
            // a full stage as straight-line MMAs (measured: a bounds check in
            // the unrolled loop slowed the weight gradients by about 7%)
            if (nkk == BK / 16) {
#pragma unroll
              for (int kk = 0; kk < BK / 16; ++kk) issue(kk);
            } else {
#pragma unroll 1
              for (int kk = 0; kk < nkk; ++kk) issue(kk);
            }
            mma_commit_pair(&sh.empty[stage], 0x3);
          }
          __syncwarp();
          if (++stage == STAGES2) stage = 0;
        }
        if (lane == 0) mma_commit_pair(&sh.tmem_full[acc], 0x3);
        __syncwarp();
        if (++acc == PAIR_ACC) acc = 0;
      }
    }
  } else if (warp == RELAY_WARP) {
    if (leader)
      relay_waits(sh, P, (int)cluster_id, (int)n_clusters, total,
                  [&](int t) { return decode_pair_tile<KGROUPED, EPI>(sh, P, t, rank); }, STAGES2,
                  PAIR_ACC, 12);
  } else {
    // ================= epilogue: warps 2..9 of both CTAs =================
    const int q = warp & 3;
    const int half = (warp - 2) >> 2;
    const int row_in_tile = q * 32 + lane;
    const uint32_t empty_base = mapa_shared(su32(&sh.tmem_empty[0]), 0);
    const uint32_t ebuf = su32(epi_buf) + (uint32_t)(warp - 2) * EPI_BOX_BYTES;
    uint32_t epi_phase = 0;  // parity of this warp's epi_load barrier
    int acc = 0;
    uint32_t acc_phase = 0;
    for (int t = cluster_id; t < total; t += n_clusters) {
      const Tile ti = decode_pair_tile<KGROUPED, EPI>(sh, P, t, rank);
      if (KGROUPED && ti.nk == 0) {
        zero_wgrad_tile(P, ti, row_in_tile, half, &tmC, ebuf);
        continue;
      }
      if (!mbar_wait(&sh.tmem_full[acc], acc_phase, sh.abort, P, 14)) { aborted = true; break; }
      tc_fence_after();
      const uint32_t t_row = tmem_base + ((uint32_t)(q * 32) << 16) + acc * BN;
      if (!drain_tile<EPI>(P, ti, t_row,
                           epi_cols(q, lane, half, EPI == EPI_SWIGLU_FWD, ti.m128 != 0), &tmC,
                           &tmD, ebuf,
                           &sh.epi_load[warp - 2], epi_phase, sh.abort)) {
        aborted = true;
        break;
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive_cluster(empty_base + acc * 8);
      if (++acc == PAIR_ACC) { acc = 0; acc_phase ^= 1; }
    }
    if (lane == 0) bulk_wait_all();  // this warp's TMA stores have landed
  }

  if (aborted || *reinterpret_cast<volatile int*>(&sh.abort)) {
    // let copies and remote arrivals already in flight land before the CTAs exit
    const uint64_t t0 = global_timer_ns();
    while (global_timer_ns() - t0 < 2000000ull) { }
  }
  pdl_launch_dependents();  // this CTA's work is done
  tc_fence_before();
  __syncthreads();
  cluster_barrier();  // neither CTA leaves while the other may still address it
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc_pair(tmem_base, PAIR_ACC * BN);
  }
}

// ---------------------------------------------------------------- SwiGLU backward, elementwise
// d_pre[r] = [dh * d act/d g | dh * d act/d u] from dh [rows, F] and the stored
// gate|up [rows, 2F] (bf16 each), 8 columns per thread with 16-byte accesses.
__global__ void __launch_bounds__(256)
glu_bwd_rows(const bf16* __restrict__ dh, const bf16* __restrict__ gu, bf16* __restrict__ d_pre,
             int64_t rows, int F, GluAct act) {
  pdl_wait();  // a dependent launch: inputs come from the kernels before
  const int per_row = F >> 3;
  const int64_t n = rows * per_row;
  for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n;
       i += (int64_t)gridDim.x * blockDim.x) {
    const int64_t r = i / per_row;
    const int f = (int)(i - r * per_row) * 8;
    float d8[8], g8[8], u8[8], dg[8], du[8];
    load_bf16x8(dh + r * F + f, d8);
    load_bf16x8(gu + r * 2 * F + f, g8);
    load_bf16x8(gu + r * 2 * F + F + f, u8);
    if (glu_is_plain(act)) {
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        const float sg = 1.f / (1.f + __expf(-g8[j]));
        dg[j] = d8[j] * u8[j] * sg * (1.f + g8[j] * (1.f - sg));
        du[j] = d8[j] * g8[j] * sg;
      }
    } else {
#pragma unroll
      for (int j = 0; j < 8; ++j) glu_bwd(g8[j], u8[j], d8[j], act, dg[j], du[j]);
    }
    store_bf16x8(d_pre + r * 2 * F + f, dg);
    store_bf16x8(d_pre + r * 2 * F + F + f, du);
  }
}

static cudaError_t launch_glu_bwd_rows(const Ctx& c, const bf16* dh, const bf16* gu, bf16* d_pre,
                                       int64_t rows, int F) {
  const int64_t n = rows * (F / 8);
  const int64_t blocks = (n + 255) / 256;
  const int64_t cap = (int64_t)c.sm_count * 16;
  launch_dependent(glu_bwd_rows, dim3((unsigned)(blocks < cap ? blocks : cap)), dim3(256), 0,
                   c.stream, dh, gu, d_pre, rows, F, c.act);
  note_launches(1);
  return cudaGetLastError();
}

// ---------------------------------------------------------------- per-expert tail maps
// For the weight gradients: per group g, copies of the two A maps (fc2: d_out,
// fc1: d_pre) whose row extent is the group's end offset, so that a TMA load
// of the group's last K block reads the following groups' rows as zeros. The
// offsets are checked as the GEMM checks them (monotone, within n_rows); the
// extent is at least 1 row.
__global__ void __launch_bounds__(256)
build_tail_maps(const __grid_constant__ CUtensorMap t0, const __grid_constant__ CUtensorMap t1,
                const int32_t* __restrict__ offsets, int G, int n_rows, CUtensorMap* out) {
  pdl_wait();  // a dependent launch: inputs come from the kernels before
  for (int g = threadIdx.x; g < G; g += blockDim.x) {
    int end = offsets ? offsets[g + 1] : n_rows;
    end = end < 1 ? 1 : (end > n_rows ? n_rows : end);
    const uint4* s0 = reinterpret_cast<const uint4*>(&t0);
    const uint4* s1 = reinterpret_cast<const uint4*>(&t1);
    uint4* d0 = reinterpret_cast<uint4*>(out + g);
    uint4* d1 = reinterpret_cast<uint4*>(out + G + g);
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      d0[i] = s0[i];
      d1[i] = s1[i];
    }
    asm volatile("tensormap.replace.tile.global_dim.global.b1024.b32 [%0], 1, %1;" ::"l"(
                     reinterpret_cast<uint64_t>(out + g)),
                 "r"(end)
                 : "memory");
    asm volatile("tensormap.replace.tile.global_dim.global.b1024.b32 [%0], 1, %1;" ::"l"(
                     reinterpret_cast<uint64_t>(out + G + g)),
                 "r"(end)
                 : "memory");
  }
  asm volatile("fence.proxy.tensormap::generic.release.gpu;" ::: "memory");
}

// ---------------------------------------------------------------- host side
static PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;
static std::mutex g_mu;

static bool get_encoder() {
  std::lock_guard<std::mutex> lk(g_mu);
  if (g_encode) return true;
  void* fn = nullptr;
  cudaDriverEntryPointQueryResult q;
  if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault,
                                       &q) != cudaSuccess ||
      q != cudaDriverEntryPointSuccess || fn == nullptr) {
    cudaGetLastError();
    return false;
  }
  g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
  return true;
}

bool make_map_bf16(CUtensorMap* m, const void* base, int64_t rows, int64_t cols, int box_rows) {
  if (!get_encoder()) return false;
  cuuint64_t gdim[2] = {(cuuint64_t)cols, (cuuint64_t)rows};
  cuuint64_t gstride[1] = {(cuuint64_t)cols * 2};
  cuuint32_t box[2] = {64u, (cuuint32_t)box_rows};
  cuuint32_t estride[2] = {1u, 1u};
  CUresult r = g_encode(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), gdim,
                        gstride, box, estride, CU_TENSOR_MAP_INTERLEAVE_NONE,
                        CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                        CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}
bool make_map_bf16_plain(CUtensorMap* m, const void* base, int64_t rows, int64_t cols,
                         int box_rows, int box_cols) {
  if (!get_encoder()) return false;
  cuuint64_t gdim[2] = {(cuuint64_t)cols, (cuuint64_t)rows};
  cuuint64_t gstride[1] = {(cuuint64_t)cols * 2};
  cuuint32_t box[2] = {(cuuint32_t)box_cols, (cuuint32_t)box_rows};
  cuuint32_t estride[2] = {1u, 1u};
  CUresult r = g_encode(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), gdim,
                        gstride, box, estride, CU_TENSOR_MAP_INTERLEAVE_NONE,
                        CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                        CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}
static bool make_map(CUtensorMap* m, const void* base, int64_t rows, int64_t cols, int box_rows) {
  return make_map_bf16(m, base, rows, cols, box_rows);
}

// Output maps for the epilogues' TMA stores: bf16 [rows, cols] with a row
// pitch of `ld` elements, 32 x 32 boxes in the 64-byte swizzle (the staging
// layout of stage_box_row). False (plain stores then) when the address or the
// pitch is not a multiple of 16 bytes.
static bool make_store_map(CUtensorMap* m, void* base, int64_t rows, int64_t cols, int64_t ld) {
  if (base == nullptr || rows <= 0 || cols <= 0 ||
      (reinterpret_cast<uintptr_t>(base) & 15) != 0 || (ld * 2) % 16 != 0 || !get_encoder())
    return false;
  cuuint64_t gdim[2] = {(cuuint64_t)cols, (cuuint64_t)rows};
  cuuint64_t gstride[1] = {(cuuint64_t)ld * 2};
  cuuint32_t box[2] = {32u, 32u};
  cuuint32_t estride[2] = {1u, 1u};
  CUresult r = g_encode(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, base, gdim, gstride, box, estride,
                        CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_64B,
                        CU_TENSOR_MAP_L2_PROMOTION_NONE, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}
// [rows, 2F] gate|up (or dg|du) as [2][rows][F]: one 32 x 16 box from each
// half per copy (32-byte swizzle, stage_box16_chunk's layout), the halves one
// after the other in shared memory (1 KB each)
static bool make_halves_map16(CUtensorMap* m, void* base, int64_t rows, int64_t F) {
  if (base == nullptr || rows <= 0 || F <= 0 || (reinterpret_cast<uintptr_t>(base) & 15) != 0 ||
      (F * 2) % 16 != 0 || !get_encoder())
    return false;
  cuuint64_t gdim[3] = {(cuuint64_t)F, (cuuint64_t)rows, 2u};
  cuuint64_t gstride[2] = {(cuuint64_t)F * 4, (cuuint64_t)F * 2};
  cuuint32_t box[3] = {16u, 32u, 2u};
  cuuint32_t estride[3] = {1u, 1u, 1u};
  CUresult r = g_encode(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, base, gdim, gstride, box, estride,
                        CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_32B,
                        CU_TENSOR_MAP_L2_PROMOTION_NONE, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}
// Weight-gradient outputs [G][rows][cols] take the staged 16-byte stores when
// their rows start on 16-byte boundaries.
static bool wgrad_rows_aligned(const void* base, int64_t cols) {
  return base != nullptr && (reinterpret_cast<uintptr_t>(base) & 15) == 0 && cols % 8 == 0;
}

constexpr size_t kSmemBytes = 1024 + (size_t)STAGES * STAGE_BYTES + EPI_BUF_BYTES + sizeof(Shared);

// ---- optional per-kernel timing (CUDA events on the launching stream)
struct KernelTiming {
  std::mutex mu;
  bool on = false;
  int device = -1;
  std::vector<cudaEvent_t> ev[kTcKinds];  // start/end pairs, in launch order
};
static KernelTiming g_timing;

static bool timing_on() { return g_timing.on; }

static void timing_mark(int kind, cudaStream_t s, bool start) {
  if (!g_timing.on) return;
  std::lock_guard<std::mutex> lk(g_timing.mu);
  int dev = -1;
  cudaGetDevice(&dev);
  if (!g_timing.on || dev != g_timing.device) return;
  cudaEvent_t e;
  if (cudaEventCreate(&e) != cudaSuccess) {
    cudaGetLastError();
    return;
  }
  cudaEventRecord(e, s);
  auto& v = g_timing.ev[kind];
  if (!start && (v.size() & 1) == 0) {  // an end without its start: drop it
    cudaEventDestroy(e);
    return;
  }
  v.push_back(e);
}

template <bool A_MN, bool B_MN, int EPI, bool GATHER = false>
static cudaError_t launch_one(const Ctx& c, const CUtensorMap& ma, const CUtensorMap& mb,
                              const CUtensorMap& mc, const CUtensorMap& md, const Params& P,
                              int kind) {
  auto kern = tc_grouped_gemm<A_MN, B_MN, EPI, GATHER>;
  static std::atomic<uint64_t> attr_set_mask{0};
  int dev = 0;
  cudaGetDevice(&dev);
  const uint64_t bit = 1ull << (dev & 63);
  if (!(attr_set_mask.load() & bit)) {
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)kSmemBytes);
    if (e != cudaSuccess) return e;
    attr_set_mask.fetch_or(bit);
  }
  cudaLaunchConfig_t cfg = {};
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;  // see pdl_wait
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.gridDim = dim3(c.sm_count);
  cfg.blockDim = dim3(NUM_THREADS);
  cfg.dynamicSmemBytes = kSmemBytes;
  cfg.stream = c.stream;
  cfg.attrs = attr;
  cfg.numAttrs = timing_on() ? 0 : 1;  // per-kernel events between launches: plain launches
  timing_mark(kind, c.stream, true);
  cudaError_t e = cudaLaunchKernelEx(&cfg, kern, ma, mb, mc, md, P);
  note_launches(1);
  timing_mark(kind, c.stream, false);
  return e;
}

constexpr size_t kSmemBytes2 = 1024 + (size_t)STAGES2 * STAGE2_BYTES + EPI_BUF_BYTES + sizeof(Shared2);

// 0: CTA pairs for long segments (default); 1: single CTAs only; 2: CTA pairs always
static std::atomic<int> g_tc_mode{0};

// CTA pairs compute 256-row tiles (a segment's last tile of at most 128 rows
// as an M = 128 tile); when the experts' segments are very short, most pair
// tiles would run at half size, so segments averaging under 128 rows stay on
// single CTAs. Measured on DeepSeek-V3-shaped layers (0 to 947 rows per expert
// at T = 8192): with the relay warp the forward at a 256-row average takes
// 5.64-5.67 ms on pairs against 5.73-5.75 ms on single CTAs; before it, a
// 128-row average (T = 4096) already ran 3.11 ms on pairs against 3.17 ms.
static bool use_pair(int G, int64_t n_rows) {
  const int mode = g_tc_mode.load();
  return mode == 2 || (mode == 0 && n_rows >= (int64_t)128 * G);
}

template <bool A_MN, bool B_MN, int EPI>
static cudaError_t launch_pair(const Ctx& c, const CUtensorMap& ma, const CUtensorMap& mb,
                               const CUtensorMap& mc, const CUtensorMap& md,
                               const CUtensorMap& ma64, const Params& P, int kind) {
  auto kern = tc_grouped_gemm_pair<A_MN, B_MN, EPI>;
  static std::atomic<uint64_t> attr_set_mask{0};
  static int max_clusters[64];
  int dev = 0;
  cudaGetDevice(&dev);
  const uint64_t bit = 1ull << (dev & 63);
  cudaLaunchConfig_t cfg = {};
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 2;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;  // see pdl_wait
  attr[1].val.programmaticStreamSerializationAllowed = 1;
  cfg.blockDim = dim3(NUM_THREADS);
  cfg.dynamicSmemBytes = kSmemBytes2;
  cfg.stream = c.stream;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  if (!(attr_set_mask.load() & bit)) {
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)kSmemBytes2);
    if (e != cudaSuccess) return e;
    cfg.gridDim = dim3(c.sm_count & ~1);
    int n = 0;
    e = cudaOccupancyMaxActiveClusters(&n, kern, &cfg);
    if (e != cudaSuccess || n <= 0) {
      cudaGetLastError();
      n = c.sm_count / 2;
    }
    max_clusters[dev & 63] = n;
    attr_set_mask.fetch_or(bit);
  }
  cfg.gridDim = dim3(2 * max_clusters[dev & 63]);
  cfg.numAttrs = timing_on() ? 1 : 2;  // per-kernel events between launches: plain launches
  timing_mark(kind, c.stream, true);
  cudaError_t e = cudaLaunchKernelEx(&cfg, kern, ma, mb, mc, md, ma64, P);
  note_launches(1);
  timing_mark(kind, c.stream, false);
  return e;
}

// M-grouped contractions (K-major A): CTA pairs or single CTAs.
template <bool B_MN, int EPI>
static cudaError_t launch_mgrouped(const Ctx& c, bool pair, const CUtensorMap& ma, const void* a,
                                   int64_t a_rows, int64_t a_cols, const CUtensorMap& mb,
                                   const CUtensorMap& mc, const CUtensorMap& md, const Params& P,
                                   int kind) {
  CUtensorMap ma64;
  if (pair) {  // its M = 128 last tiles load 64 A rows per CTA
    if (!make_map(&ma64, a, a_rows, a_cols, 64)) return cudaErrorInvalidValue;
    return launch_pair<false, B_MN, EPI>(c, ma, mb, mc, md, ma64, P, kind);
  }
  return launch_one<false, B_MN, EPI>(c, ma, mb, mc, md, P, kind);
}

// M = 128 last tiles on CTA pairs (with 64-row A loads): measured 2% faster
// on the Mixtral-sized step and about 1% on the fine-grained and Zipf-skewed
// ones against 256-row tiles throughout.
static int m128_tails_for(int) { return 1; }

static Params base_params(const Ctx& c, int G, int64_t n_rows, const int32_t* offsets) {
  Params P{};
  P.G = G;
  P.n_rows = (int)n_rows;
  P.offsets = offsets;
  P.status = c.status;
  P.timeout_ns = c.timeout_ns;
  P.act = c.act;
  return P;
}

}  // namespace tc

bool tc_available() { return tc::get_encoder(); }

size_t tc_grouped_ws_bytes(int) { return 0; }

size_t tc_tail_maps_bytes(int n_groups) { return (size_t)2 * n_groups * sizeof(CUtensorMap) + 128; }

int tc_set_mode(int mode) { return tc::g_tc_mode.exchange(mode); }

int tc_timing_enable(int on) {
  using namespace tc;
  std::lock_guard<std::mutex> lk(g_timing.mu);
  if (!on) {  // stop recording; keep what was recorded for tc_timing_read
    g_timing.on = false;
    return MOE_OK;
  }
  for (int k = 0; k < kTcKinds; ++k) {
    for (cudaEvent_t e : g_timing.ev[k]) cudaEventDestroy(e);
    g_timing.ev[k].clear();
  }
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess) {
    cudaGetLastError();
    g_timing.on = false;
    return MOE_ERR_NO_DEVICE;
  }
  g_timing.device = dev;
  g_timing.on = true;
  return MOE_OK;
}

int tc_timing_read(float* ms_total, int32_t* launches) {
  using namespace tc;
  std::lock_guard<std::mutex> lk(g_timing.mu);
  for (int k = 0; k < kTcKinds; ++k) {
    float tot = 0.f;
    int n = 0;
    auto& v = g_timing.ev[k];
    for (size_t i = 0; i + 1 < v.size(); i += 2) {
      if (cudaEventSynchronize(v[i + 1]) != cudaSuccess) return MOE_ERR_CUDA;
      float ms = 0.f;
      if (cudaEventElapsedTime(&ms, v[i], v[i + 1]) != cudaSuccess) return MOE_ERR_CUDA;
      tot += ms;
      ++n;
    }
    if (ms_total) ms_total[k] = tot;
    if (launches) launches[k] = n;
  }
  return MOE_OK;
}

cudaError_t launch_tc_grouped_swiglu_fwd(const Ctx& c, int G, int64_t n_rows, int F, int d,
                                         const int32_t* offsets, const void* x_rows,
                                         const void* w1, const void* w2, void* pre_gu, void* h,
                                         void* out, void*, int* err) {
  using namespace tc;
  *err = MOE_OK;
  if (n_rows == 0) return cudaSuccess;
  CUtensorMap mA, mB;
  const bool pair = use_pair(G, n_rows);
  // fc1: A = x_rows [n_rows, d] (K-major), B = W1 [G*2F, d] (K-major; single
  // CTAs load 128 gate and 128 up rows, a CTA of a pair 64 of each)
  if (!make_map(&mA, x_rows, n_rows, d, 128) ||
      !make_map(&mB, w1, (int64_t)G * 2 * F, d, pair ? 64 : 128)) {
    *err = MOE_ERR_CUDA;
    return cudaSuccess;
  }
  Params P = base_params(c, G, n_rows, offsets);
  P.K = d;
  P.m128_tails = m128_tails_for(P.K);
  P.F = F;
  P.NT = (F + BN / 2 - 1) / (BN / 2);
  P.out0 = static_cast<bf16*>(h);
  P.ld0 = F;
  P.out1 = static_cast<bf16*>(pre_gu);
  // h and gate|up stored through the TMA unit (both maps, or neither)
  CUtensorMap mH, mGU;
  P.tma_out = make_store_map(&mH, h, n_rows, F, F) &&
              (pre_gu == nullptr || make_store_map(&mGU, pre_gu, n_rows, 2 * F, 2 * F));
  if (!P.tma_out) mH = mA;
  if (!P.tma_out || pre_gu == nullptr) mGU = mH;
  cudaError_t e = launch_mgrouped<false, EPI_SWIGLU_FWD>(c, pair, mA, x_rows, n_rows, d, mB, mH,
                                                         mGU, P, kFc1Fwd);
  if (e != cudaSuccess) return e;
  // fc2: A = h [n_rows, F], B = W2 [G*d, F] (K-major, 256-row boxes)
  if (!make_map(&mA, h, n_rows, F, 128) || !make_map(&mB, w2, (int64_t)G * d, F, pair ? 128 : 256)) {
    *err = MOE_ERR_CUDA;
    return cudaSuccess;
  }
  Params Q = base_params(c, G, n_rows, offsets);
  Q.K = F;
  Q.m128_tails = m128_tails_for(Q.K);
  Q.N_out = d;
  Q.NT = (d + BN - 1) / BN;
  Q.b_group_rows = d;
  Q.out0 = static_cast<bf16*>(out);
  Q.ld0 = d;
  CUtensorMap mC;
  Q.tma_out = make_store_map(&mC, out, n_rows, d, d);
  if (!Q.tma_out) mC = mA;
  return launch_mgrouped<false, EPI_STORE>(c, pair, mA, h, n_rows, F, mB, mC, mC, Q, kFc2Fwd);
}

cudaError_t launch_tc_grouped_swiglu_fwd_gather(const Ctx& c, int G, int64_t n_rows, int F, int d,
                                                const int32_t* offsets, const void* x,
                                                int64_t x_rows, const int32_t* src_rows,
                                                const void* w1, const void* w2, void* pre_gu,
                                                void* h, void* out, int* err) {
  using namespace tc;
  *err = MOE_OK;
  if (n_rows == 0) return cudaSuccess;
  // fc1 on single CTAs with the A rows gathered from x; B = W1 [G*2F, d]
  CUtensorMap mB;
  if (!make_map(&mB, w1, (int64_t)G * 2 * F, d, 128)) {
    *err = MOE_ERR_CUDA;
    return cudaSuccess;
  }
  Params P = base_params(c, G, n_rows, offsets);
  P.K = d;
  P.F = F;
  P.NT = (F + BN / 2 - 1) / (BN / 2);
  P.out0 = static_cast<bf16*>(h);
  P.ld0 = F;
  P.out1 = static_cast<bf16*>(pre_gu);
  P.a_rows = static_cast<const bf16*>(x);
  P.a_src = src_rows;
  P.a_src_rows = (int)x_rows;
  CUtensorMap mH, mGU;
  P.tma_out = make_store_map(&mH, h, n_rows, F, F) &&
              (pre_gu == nullptr || make_store_map(&mGU, pre_gu, n_rows, 2 * F, 2 * F));
  if (!P.tma_out) mH = mB;
  if (!P.tma_out || pre_gu == nullptr) mGU = mH;
  cudaError_t e = launch_one<false, false, EPI_SWIGLU_FWD, true>(c, mB, mB, mH, mGU, P, kFc1Fwd);
  if (e != cudaSuccess) return e;
  // fc2 as in the plain forward: A = h [n_rows, F]
  CUtensorMap mA;
  const bool pair = use_pair(G, n_rows);
  if (!make_map(&mA, h, n_rows, F, 128) || !make_map(&mB, w2, (int64_t)G * d, F, pair ? 128 : 256)) {
    *err = MOE_ERR_CUDA;
    return cudaSuccess;
  }
  Params Q = base_params(c, G, n_rows, offsets);
  Q.K = F;
  Q.m128_tails = m128_tails_for(Q.K);
  Q.N_out = d;
  Q.NT = (d + BN - 1) / BN;
  Q.b_group_rows = d;
  Q.out0 = static_cast<bf16*>(out);
  Q.ld0 = d;
  CUtensorMap mC;
  Q.tma_out = make_store_map(&mC, out, n_rows, d, d);
  if (!Q.tma_out) mC = mA;
  return launch_mgrouped<false, EPI_STORE>(c, pair, mA, h, n_rows, F, mB, mC, mC, Q, kFc2Fwd);
}

cudaError_t launch_tc_grouped_swiglu_bwd(const Ctx& c, int G, int64_t n_rows, int F, int d,
                                         const int32_t* offsets, const void* x_rows,
                                         const void* w1, const void* w2, const void* pre_gu,
                                         const void* h, const void* d_out, void* d_pre,
                                         void* dx_rows, void* dw1, void* dw2, void* ws,
                                         size_t ws_bytes, int* err) {
  using namespace tc;
  *err = MOE_OK;
  CUtensorMap mA, mB, mC;
  cudaError_t e;
  // the weight gradients' per-expert tail maps sit at the end of the workspace
  const int mode = g_tc_mode.load();
  const bool wpair = mode != 1;  // weight gradients: CTA pairs unless single-CTA
  CUtensorMap* tail_maps = nullptr;
  if (n_rows > 0 && wpair && ws != nullptr && ws_bytes >= tc_tail_maps_bytes(G)) {
    const uintptr_t end = reinterpret_cast<uintptr_t>(ws) + ws_bytes;
    tail_maps = reinterpret_cast<CUtensorMap*>((end - 2 * (size_t)G * sizeof(CUtensorMap)) &
                                               ~(uintptr_t)127);
    ws_bytes -= tc_tail_maps_bytes(G);
  }
  if (n_rows > 0) {
    // fc2 dgrad: A = d_out [n_rows, d] K-major; B = W2 [G*d, F] MN-major. With a
    // short K (d < 4096) a tile's MMAs do not hide the SwiGLU-backward
    // epilogue, so the GEMM stores dh (bf16) and an elementwise pass applies
    // the derivative; with d >= 4096 the derivative runs in the epilogue.
    const size_t dh_bytes = ((size_t)n_rows * F * 2 + 255) & ~(size_t)255;
    const bool split = d < 4096 && ws != nullptr && ws_bytes >= dh_bytes;
    if (!make_map(&mA, d_out, n_rows, d, 128) || !make_map(&mB, w2, (int64_t)G * d, F, 64)) {
      *err = MOE_ERR_CUDA;
      return cudaSuccess;
    }
    Params P = base_params(c, G, n_rows, offsets);
    P.K = d;
    P.m128_tails = m128_tails_for(P.K);
    P.F = F;
    P.N_out = F;
    P.NT = (F + BN - 1) / BN;
    P.b_group_rows = d;
    const bool pair = use_pair(G, n_rows);
    if (split) {
      P.out0 = static_cast<bf16*>(ws);
      P.ld0 = F;
      P.tma_out = make_store_map(&mC, ws, n_rows, F, F);
      if (!P.tma_out) mC = mA;
      e = launch_mgrouped<true, EPI_STORE>(c, pair, mA, d_out, n_rows, d, mB, mC, mC, P,
                                           kFc2Dgrad);
      if (e != cudaSuccess) return e;
      e = launch_glu_bwd_rows(c, static_cast<const bf16*>(ws), static_cast<const bf16*>(pre_gu),
                              static_cast<bf16*>(d_pre), n_rows, F);
    } else {
      P.out0 = static_cast<bf16*>(d_pre);
      P.aux_in = static_cast<const bf16*>(pre_gu);
      // d_pre out (tmC) and gate|up in (tmD) as 32 x 16 boxes of both halves
      CUtensorMap mGU;
      P.tma_out = make_halves_map16(&mC, d_pre, n_rows, F) &&
                  make_halves_map16(&mGU, const_cast<void*>(pre_gu), n_rows, F);
      if (!P.tma_out) mC = mGU = mA;
      e = launch_mgrouped<true, EPI_SWIGLU_BWD>(c, pair, mA, d_out, n_rows, d, mB, mC, mGU, P,
                                                kFc2Dgrad);
    }
    if (e != cudaSuccess) return e;
    // fc1 dgrad: A = d_pre [n_rows, 2F] K-major; B = W1 [G*2F, d] MN-major
    if (!make_map(&mA, d_pre, n_rows, 2 * F, 128) || !make_map(&mB, w1, (int64_t)G * 2 * F, d, 64)) {
      *err = MOE_ERR_CUDA;
      return cudaSuccess;
    }
    Params Q = base_params(c, G, n_rows, offsets);
    Q.K = 2 * F;
    Q.m128_tails = m128_tails_for(Q.K);
    Q.N_out = d;
    Q.NT = (d + BN - 1) / BN;
    Q.b_group_rows = 2 * F;
    Q.out0 = static_cast<bf16*>(dx_rows);
    Q.ld0 = d;
    Q.tma_out = make_store_map(&mC, dx_rows, n_rows, d, d);
    if (!Q.tma_out) mC = mA;
    e = launch_mgrouped<true, EPI_STORE>(c, pair, mA, d_pre, n_rows, 2 * F, mB, mC, mC, Q,
                                         kFc1Dgrad);
    if (e != cudaSuccess) return e;
  }
  // fc2 wgrad: dW2_g [d, F] = d_outᵀ h : A = d_out [n_rows, d] MN-major, B = h [n_rows, F] MN-major
  // (with no rows at all, 1-row maps are never read: every group is empty)
  const int64_t mr = n_rows > 0 ? n_rows : 1;
  if (!make_map(&mA, n_rows > 0 ? d_out : w2, mr, d, 64) ||
      !make_map(&mB, n_rows > 0 ? h : w2, mr, F, 64)) {
    *err = MOE_ERR_CUDA;
    return cudaSuccess;
  }
  if (tail_maps != nullptr) {
    CUtensorMap mA1;  // fc1 wgrad's A: d_pre [n_rows, 2F]
    if (!make_map(&mA1, d_pre, mr, 2 * F, 64)) {
      *err = MOE_ERR_CUDA;
      return cudaSuccess;
    }
    launch_dependent(build_tail_maps, dim3(1), dim3(256), 0, c.stream, mA, mA1, offsets, G,
                     (int)n_rows, tail_maps);
    note_launches(1);
    e = cudaGetLastError();
    if (e != cudaSuccess) return e;
  }
  Params R = base_params(c, G, n_rows, offsets);
  R.M_out = d;
  R.N_out = F;
  R.tail_maps = tail_maps;
  R.MT = wpair ? (d + 2 * BM - 1) / (2 * BM) : (d + BM - 1) / BM;
  R.NT = (F + BN - 1) / BN;
  R.out0 = static_cast<bf16*>(dw2);
  R.tma_out = wgrad_rows_aligned(dw2, F);
  e = wpair ? launch_pair<true, true, EPI_WGRAD>(c, mA, mB, mA, mA, mA, R, kFc2Wgrad)
            : launch_one<true, true, EPI_WGRAD>(c, mA, mB, mA, mA, R, kFc2Wgrad);
  if (e != cudaSuccess) return e;
  // fc1 wgrad: dW1_g [2F, d] = d_preᵀ x : A = d_pre [n_rows, 2F] MN-major, B = x_rows MN-major
  if (!make_map(&mA, n_rows > 0 ? d_pre : w1, mr, 2 * F, 64) ||
      !make_map(&mB, n_rows > 0 ? x_rows : w1, mr, d, 64)) {
    *err = MOE_ERR_CUDA;
    return cudaSuccess;
  }
  Params S = base_params(c, G, n_rows, offsets);
  S.M_out = 2 * F;
  S.N_out = d;
  S.tail_maps = tail_maps != nullptr ? tail_maps + G : nullptr;
  S.MT = wpair ? (2 * F + 2 * BM - 1) / (2 * BM) : (2 * F + BM - 1) / BM;
  S.NT = (d + BN - 1) / BN;
  S.out0 = static_cast<bf16*>(dw1);
  S.tma_out = wgrad_rows_aligned(dw1, d);
  return wpair ? launch_pair<true, true, EPI_WGRAD>(c, mA, mB, mA, mA, mA, S, kFc1Wgrad)
               : launch_one<true, true, EPI_WGRAD>(c, mA, mB, mA, mA, S, kFc1Wgrad);
}

}  // namespace moe
