// The extern "C" entry points declared in include/moe.h: argument checks,
// the device status word, workspace sizing, and the order in which each call
// launches its kernels on the caller's stream.
#include <algorithm>
#include <atomic>
#include <cmath>
#include <cstdio>
#include <mutex>

#include "common.cuh"
#include "internal.h"

namespace moe {

// status[0] = first error code, status[1] = detail, status[2] = a flag nothing sets
__device__ int g_status[4];

static std::atomic<uint64_t> g_timeout_ns{2000000000ull};
static std::atomic<uint64_t> g_launches{0};
static std::atomic<int> g_gemm_impl{MOE_GEMM_AUTO};

static bool use_tc(int dt) {
  return dt == kBF16 && g_gemm_impl.load() == MOE_GEMM_AUTO && tc_available();
}

void note_launches(int n) { g_launches.fetch_add((uint64_t)n, std::memory_order_relaxed); }
uint64_t launches_so_far() { return g_launches.load(std::memory_order_relaxed); }

constexpr int kMaxDevices = 64;
static std::mutex g_dev_mu;
static int* g_status_ptr[kMaxDevices];
static int g_sm_count[kMaxDevices];

static int make_ctx(cudaStream_t stream, Ctx* c) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) {
    cudaGetLastError();
    return MOE_ERR_NO_DEVICE;
  }
  std::lock_guard<std::mutex> lk(g_dev_mu);
  if (g_status_ptr[dev] == nullptr) {
    int major = 0, minor = 0, sms = 0;
    if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) {
      cudaGetLastError();
      return MOE_ERR_NO_DEVICE;
    }
    if (major != 10 || minor != 3) return MOE_ERR_NO_DEVICE;  // built for sm_103a only
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_status) != cudaSuccess) {
      cudaGetLastError();
      return MOE_ERR_CUDA;
    }
    g_sm_count[dev] = sms;
    g_status_ptr[dev] = static_cast<int*>(p);
  }
  c->stream = stream;
  c->status = g_status_ptr[dev];
  c->timeout_ns = g_timeout_ns.load();
  c->sm_count = g_sm_count[dev];
  c->act = GluAct{MOE_ACT_SWIGLU, 0.f, 0.f, 0.f, 0.f};
  return MOE_OK;
}


static bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

static int check_cfg(const moe_cfg* cfg) {
  if (cfg == nullptr) return MOE_ERR_INVALID_ARG;
  if (cfg->T < 0 || cfg->d <= 0 || cfg->E <= 0 || cfg->k <= 0 || cfg->F <= 0 ||
      cfg->F_shared < 0)
    return MOE_ERR_INVALID_ARG;
  if (cfg->score_fn < MOE_SCORE_SOFTMAX || cfg->score_fn > MOE_SCORE_SOFTMAX_PRE)
    return MOE_ERR_INVALID_ARG;
  if (cfg->act_dtype != MOE_F32 && cfg->act_dtype != MOE_BF16) return MOE_ERR_INVALID_ARG;
  if (cfg->k > cfg->E) return MOE_ERR_INVALID_ARG;
  // The Ultimate MoE Training Handbook, §3.1 "Output scale": softmax over a
  // single chosen logit is always 1, so top-1 softmax with renormalisation
  // gives the router no gradient and is refused.
  if (cfg->score_fn == MOE_SCORE_SOFTMAX && cfg->k == 1) return MOE_ERR_INVALID_ARG;
  if (cfg->E > kMaxE || cfg->k > kMaxK) return MOE_ERR_UNSUPPORTED;
  if ((cfg->d & 7) || (cfg->F & 7) || (cfg->F_shared & 7)) return MOE_ERR_ALIGN;
  if (cfg->T * (int64_t)cfg->k >= (int64_t)0x7fffffff) return MOE_ERR_UNSUPPORTED;
  // expert activation (Handbook §3.4 "Activation"): the SwiGLU clamp value
  // must be finite and > 0 with a zero linear offset; SiTU needs a gate scale
  switch (cfg->act_fn) {
    case MOE_ACT_SWIGLU: break;
    case MOE_ACT_SWIGLU_CLAMP:
      if (!(std::isfinite(cfg->act_clamp) && cfg->act_clamp > 0.f) ||
          cfg->glu_linear_offset != 0.f)
        return MOE_ERR_INVALID_ARG;
      break;
    case MOE_ACT_SITU_GLU:
      if (!(std::isfinite(cfg->act_gate_scale) && cfg->act_gate_scale > 0.f) ||
          !(std::isfinite(cfg->act_linear_scale) && cfg->act_linear_scale >= 0.f))
        return MOE_ERR_INVALID_ARG;
      break;
    default: return MOE_ERR_INVALID_ARG;
  }
  if (!std::isfinite(cfg->glu_linear_offset)) return MOE_ERR_INVALID_ARG;
  return MOE_OK;
}
static_assert(sizeof(moe_cfg) == 64, "moe_cfg layout");

static int act_size(const moe_cfg& cfg) { return cfg.act_dtype == MOE_BF16 ? 2 : 4; }

#define MOE_REQUIRE(cond, code) \
  do {                           \
    if (!(cond)) return (code);  \
  } while (0)
#define MOE_PTR(p) MOE_REQUIRE((p) != nullptr, MOE_ERR_INVALID_ARG); MOE_REQUIRE(aligned16(p), MOE_ERR_ALIGN)
#define MOE_OPT_PTR(p) MOE_REQUIRE((p) == nullptr || aligned16(p), MOE_ERR_ALIGN)
#define MOE_CHECK_CFG(cfg)               \
  do {                                   \
    const int _rc = check_cfg(cfg);      \
    if (_rc != MOE_OK) return _rc;       \
  } while (0)
#define MOE_CTX(stream, ctx)                                   \
  Ctx ctx;                                                     \
  do {                                                         \
    const int _rc = make_ctx((cudaStream_t)(stream), &ctx);    \
    if (_rc != MOE_OK) return _rc;                             \
  } while (0)
// the CUDA error behind the calling thread's last MOE_ERR_CUDA
static thread_local cudaError_t g_last_cuda_error = cudaSuccess;
static int cuda_failed(cudaError_t e) {
  g_last_cuda_error = e;
  cudaGetLastError();  // clear a non-sticky error so later calls can run
  return MOE_ERR_CUDA;
}

#define MOE_LAUNCH(expr)                               \
  do {                                                 \
    const cudaError_t _e = (expr);                     \
    if (_e != cudaSuccess) return cuda_failed(_e);     \
  } while (0)

// K (token) slices of the dW_r reduction; partials [S][E][d] fp32 in the workspace
static int route_bwd_splits(const moe_cfg& cfg) {
  // few experts: slices of >= 32 tokens, up to 128 of them (enough CTAs of the
  // column-blocked kernel to keep every SM's loads in flight)
  int64_t s = (cfg.E <= 16) ? (cfg.T + 31) / 32 : (cfg.T + 511) / 512;
  const int64_t cap = (cfg.E <= 16) ? 128 : 32;
  if (s < 1) s = 1;
  if (s > cap) s = cap;
  return (int)s;
}

static size_t round256(size_t n) { return (n + 255) & ~(size_t)255; }

static size_t grouped_fwd_ws(const moe_cfg& cfg) {
  const size_t es = (size_t)act_size(cfg);
  size_t rows_r = (size_t)cfg.T * cfg.k, rows_s = (size_t)cfg.T;
  size_t need = round256(rows_r * 2 * cfg.F * es);  // gate|up when the caller passes none
  if (cfg.F_shared > 0) {
    const size_t s = round256(rows_s * 2 * cfg.F_shared * es);
    if (s > need) need = s;
  }
  return need + round256(tc_grouped_ws_bytes(cfg.E));
}

static size_t grouped_bwd_ws(const moe_cfg& cfg) {
  size_t rows_r = (size_t)cfg.T * cfg.k, rows_s = (size_t)cfg.T;
  size_t need = round256(rows_r * cfg.F * sizeof(float));  // dh in fp32
  if (cfg.F_shared > 0) {
    const size_t s = round256(rows_s * cfg.F_shared * sizeof(float));
    if (s > need) need = s;
  }
  return need + round256(tc_grouped_ws_bytes(cfg.E)) + round256(tc_tail_maps_bytes(cfg.E));
}

static size_t route_bwd_ws(const moe_cfg& cfg) {
  const size_t simt = round256((size_t)route_bwd_splits(cfg) * cfg.E * cfg.d * sizeof(float));
  return router_bwd_tc_shape(cfg) ? std::max(simt, round256(router_bwd_tc_ws_bytes(cfg))) : simt;
}

static size_t shared_gate_bwd_ws(const moe_cfg& cfg) {
  moe_cfg one = cfg;
  one.E = 1;
  return round256((size_t)route_bwd_splits(one) * cfg.d * sizeof(float));
}

}  // namespace moe

using namespace moe;

extern "C" {

int moe_check_cfg(const moe_cfg* cfg) { return check_cfg(cfg); }

const char* moe_version(void) { return "libmoe 0.1 sm_103a"; }

const char* moe_status_string(int status) {
  switch (status) {
    case MOE_OK: return "ok";
    case MOE_ERR_INVALID_ARG: return "invalid argument or refused configuration";
    case MOE_ERR_UNSUPPORTED: return "unsupported size (E <= 256, k <= 8, T*k < 2^31)";
    case MOE_ERR_ALIGN: return "row or pointer not 16-byte aligned (d, F must be multiples of 8)";
    case MOE_ERR_CUDA: return "CUDA runtime call or kernel launch failed";
    case MOE_ERR_TIMEOUT: return "a bounded device wait ran out of time";
    case MOE_ERR_DEVICE_INDEX: return "device saw an index or offset out of range";
    case MOE_ERR_WORKSPACE: return "workspace smaller than moe_workspace_bytes()";
    case MOE_ERR_NO_DEVICE: return "no usable sm_103 device";
    default: return "unknown status";
  }
}

uint64_t moe_set_wait_timeout_ns(uint64_t ns) { return g_timeout_ns.exchange(ns); }

uint64_t moe_launch_count(void) { return launches_so_far(); }

int moe_kernel_timing(int enable) { return tc_timing_enable(enable); }

int moe_kernel_times(float* ms_total, int32_t* launches) {
  return tc_timing_read(ms_total, launches);
}

int moe_set_grouped_gemm_impl(int impl) {
  if (impl != MOE_GEMM_AUTO && impl != MOE_GEMM_CUDA_CORES && impl != MOE_GEMM_TC_SINGLE_CTA &&
      impl != MOE_GEMM_TC_PAIRS)
    return MOE_ERR_INVALID_ARG;
  static std::atomic<int> g_public{MOE_GEMM_AUTO};
  tc_set_mode(impl == MOE_GEMM_TC_SINGLE_CTA ? 1 : impl == MOE_GEMM_TC_PAIRS ? 2 : 0);
  g_gemm_impl.store(impl == MOE_GEMM_CUDA_CORES ? MOE_GEMM_CUDA_CORES : MOE_GEMM_AUTO);
  return g_public.exchange(impl);
}

int moe_set_router_impl(int impl) {
  if (impl != MOE_ROUTER_AUTO && impl != MOE_ROUTER_CUDA_CORES) return MOE_ERR_INVALID_ARG;
  return router_set_impl(impl == MOE_ROUTER_CUDA_CORES ? 1 : 0);
}

int moe_set_router_fold(int fold_k) {
  if (fold_k < 16 || fold_k > 4096 || fold_k % 16 != 0) return MOE_ERR_INVALID_ARG;
  return router_set_fold(fold_k);
}

const char* moe_last_cuda_error(void) {
  static thread_local char buf[256];
  if (g_last_cuda_error == cudaSuccess) return "";
  snprintf(buf, sizeof(buf), "%s: %s", cudaGetErrorName(g_last_cuda_error),
           cudaGetErrorString(g_last_cuda_error));
  return buf;
}

int moe_router_uses_tensor_cores(const moe_cfg* cfg) {
  if (check_cfg(cfg) != MOE_OK) return 0;
  return router_tc_eligible(*cfg) ? 1 : 0;
}

int moe_router_bwd_uses_tensor_cores(const moe_cfg* cfg) {
  if (check_cfg(cfg) != MOE_OK) return 0;
  return router_bwd_tc_eligible(*cfg) ? 1 : 0;
}

int moe_last_device_status(moe_stream_t stream, int32_t* detail) {
  MOE_CTX(stream, c);
  MOE_LAUNCH(cudaStreamSynchronize(c.stream));
  int h[2] = {0, 0};
  MOE_LAUNCH(cudaMemcpy(h, c.status, sizeof(h), cudaMemcpyDeviceToHost));
  MOE_LAUNCH(cudaMemset(c.status, 0, 2 * sizeof(int)));
  if (detail) *detail = h[1];
  return h[0];
}

size_t moe_workspace_bytes(const moe_cfg* cfg, int which) {
  if (check_cfg(cfg) != MOE_OK) return 0;
  switch (which) {
    case MOE_WS_PERMUTE: return permute_ws_bytes(*cfg);
    case MOE_WS_GROUPED: return grouped_fwd_ws(*cfg);
    case MOE_WS_GROUPED_BWD: return grouped_bwd_ws(*cfg);
    case MOE_WS_AUX: return aux_ws_bytes(*cfg);
    case MOE_WS_ROUTE_BWD: return route_bwd_ws(*cfg);
    case MOE_WS_ROUTE: return router_ws_bytes(*cfg);
    case MOE_WS_Z_LOSS: return z_loss_ws_bytes(*cfg);
    case MOE_WS_SHARED_GATE_BWD: return shared_gate_bwd_ws(*cfg);
    default: return 0;
  }
}

int moe_route_topk(const moe_cfg* cfg, const void* x, const float* w_router,
                   const float* logit_bias, const float* sel_bias, float* logits, int32_t* idx,
                   float* w, void* ws, size_t ws_bytes, moe_stream_t stream) {
  MOE_CHECK_CFG(cfg);
  if (sel_bias != nullptr && !score_takes_bias(cfg->score_fn)) return MOE_ERR_INVALID_ARG;
  if (cfg->T == 0) return MOE_OK;
  MOE_PTR(x); MOE_PTR(w_router); MOE_PTR(logits); MOE_PTR(idx); MOE_PTR(w);
  MOE_REQUIRE(logit_bias == nullptr || (reinterpret_cast<uintptr_t>(logit_bias) & 3u) == 0, MOE_ERR_ALIGN);
  MOE_REQUIRE(sel_bias == nullptr || (reinterpret_cast<uintptr_t>(sel_bias) & 3u) == 0, MOE_ERR_ALIGN);
  const size_t need = router_ws_bytes(*cfg);
  MOE_REQUIRE(ws_bytes >= need, MOE_ERR_WORKSPACE);
  if (need > 0) { MOE_PTR(ws); }
  MOE_CTX(stream, c);
  MOE_LAUNCH(launch_router_logits(c, *cfg, x, w_router, logit_bias, logits,
                                  need > 0 ? ws : nullptr));
  MOE_LAUNCH(launch_router_topk(c, *cfg, logits, sel_bias, idx, w));
  return MOE_OK;
}

int moe_route_near_ties(const moe_cfg* cfg, const float* logits, const float* sel_bias,
                        float band, int32_t* count, moe_stream_t stream) {
  MOE_CHECK_CFG(cfg);
  if (sel_bias != nullptr && !score_takes_bias(cfg->score_fn)) return MOE_ERR_INVALID_ARG;
  MOE_REQUIRE(std::isfinite(band) && band >= 0.f, MOE_ERR_INVALID_ARG);
  MOE_REQUIRE(count != nullptr && (reinterpret_cast<uintptr_t>(count) & 3u) == 0, MOE_ERR_ALIGN);
  if (cfg->T > 0) { MOE_PTR(logits); }
  MOE_REQUIRE(sel_bias == nullptr || (reinterpret_cast<uintptr_t>(sel_bias) & 3u) == 0, MOE_ERR_ALIGN);
  MOE_CTX(stream, c);
  MOE_LAUNCH(launch_router_near_ties(c, *cfg, logits, sel_bias, band, count));
  return MOE_OK;
}

int moe_permute(const moe_cfg* cfg, const void* x, const int32_t* idx, int32_t* counts,
                int32_t* offsets, int32_t* row_of, int32_t* src_tok, void* x_perm, void* ws,
                size_t ws_bytes, moe_stream_t stream) {
  MOE_CHECK_CFG(cfg);
  MOE_PTR(counts); MOE_PTR(offsets);
  if (cfg->T > 0) {
    MOE_PTR(idx); MOE_PTR(row_of); MOE_PTR(src_tok); MOE_PTR(ws);
    MOE_OPT_PTR(x_perm);  // NULL: the index outputs only, no row copy
    if (x_perm != nullptr) { MOE_PTR(x); }
  }
  MOE_REQUIRE(ws_bytes >= permute_ws_bytes(*cfg), MOE_ERR_WORKSPACE);
  MOE_CTX(stream, c);
  MOE_LAUNCH(launch_permute(c, *cfg, x, idx, counts, offsets, row_of, src_tok, x_perm, ws));
  return MOE_OK;
}

int moe_grouped_swiglu(const moe_cfg* cfg, int32_t n_groups, int64_t n_rows, int32_t F,
                       const int32_t* offsets, const void* x_rows, const void* w1,
                       const void* w2, void* pre_gu, void* h, void* out, void* ws,
                       size_t ws_bytes, moe_stream_t stream) {
  MOE_CHECK_CFG(cfg);
  MOE_REQUIRE(n_groups >= 1 && n_groups <= kMaxE && n_rows >= 0 && F > 0, MOE_ERR_INVALID_ARG);
  MOE_REQUIRE((F & 7) == 0, MOE_ERR_ALIGN);
  MOE_REQUIRE(offsets != nullptr || n_groups == 1, MOE_ERR_INVALID_ARG);
  MOE_REQUIRE(n_rows < (int64_t)0x7fffffff, MOE_ERR_UNSUPPORTED);
  MOE_PTR(w1); MOE_PTR(w2); MOE_OPT_PTR(pre_gu); MOE_OPT_PTR(offsets);
  if (n_rows > 0) { MOE_PTR(x_rows); MOE_PTR(h); MOE_PTR(out); }
  MOE_CTX(stream, c);
  c.act = glu_act_of(*cfg);
  if (n_rows == 0) return MOE_OK;
  const int dt = cfg->act_dtype == MOE_BF16 ? kBF16 : kF32;
  const int d = cfg->d;
  if (use_tc(dt)) {
    MOE_REQUIRE(ws_bytes >= round256(tc_grouped_ws_bytes(n_groups)), MOE_ERR_WORKSPACE);
    MOE_REQUIRE(ws != nullptr || tc_grouped_ws_bytes(n_groups) == 0, MOE_ERR_INVALID_ARG);
    int err = MOE_OK;
    MOE_LAUNCH(launch_tc_grouped_swiglu_fwd(c, n_groups, n_rows, F, d, offsets, x_rows, w1, w2,
                                            pre_gu, h, out, ws, &err));
    return err;
  }
  void* pre = pre_gu;
  if (pre == nullptr) {
    MOE_PTR(ws);
    MOE_REQUIRE(ws_bytes >= round256((size_t)n_rows * 2 * F * act_size(*cfg)), MOE_ERR_WORKSPACE);
    pre = ws;
  }
  SimtGemm g1{};
  g1.mode = kGroupM; g1.M = (int)n_rows; g1.N = 2 * F; g1.K = d;
  g1.dtA = g1.dtB = g1.dtC = dt;
  g1.A = x_rows; g1.a_sm = d; g1.a_sk = 1; g1.a_sg = 0;
  g1.B = w1; g1.b_sn = d; g1.b_sk = 1; g1.b_sg = (int64_t)2 * F * d;
  g1.C = pre; g1.c_sm = 2 * F; g1.c_sg = 0;
  g1.offsets = offsets; g1.n_groups = n_groups; g1.alpha = 1.f;
  MOE_LAUNCH(launch_simt_gemm(c, g1));
  MOE_LAUNCH(launch_swiglu_fwd_elem(c, dt, pre, h, n_rows, F));  // c.act
  SimtGemm g2{};
  g2.mode = kGroupM; g2.M = (int)n_rows; g2.N = d; g2.K = F;
  g2.dtA = g2.dtB = g2.dtC = dt;
  g2.A = h; g2.a_sm = F; g2.a_sk = 1;
  g2.B = w2; g2.b_sn = F; g2.b_sk = 1; g2.b_sg = (int64_t)d * F;
  g2.C = out; g2.c_sm = d;
  g2.offsets = offsets; g2.n_groups = n_groups; g2.alpha = 1.f;
  MOE_LAUNCH(launch_simt_gemm(c, g2));
  return MOE_OK;
}

int moe_grouped_swiglu_gather(const moe_cfg* cfg, int32_t n_groups, int64_t n_rows, int32_t F,
                              const int32_t* offsets, const void* x, int64_t x_rows,
                              const int32_t* src_rows, const void* w1, const void* w2,
                              void* pre_gu, void* h, void* out, moe_stream_t stream) {
  MOE_CHECK_CFG(cfg);
  MOE_REQUIRE(n_groups >= 1 && n_groups <= kMaxE && n_rows >= 0 && F > 0 && x_rows >= 0,
              MOE_ERR_INVALID_ARG);
  MOE_REQUIRE((F & 7) == 0, MOE_ERR_ALIGN);
  MOE_REQUIRE(offsets != nullptr || n_groups == 1, MOE_ERR_INVALID_ARG);
  MOE_REQUIRE(n_rows < (int64_t)0x7fffffff && x_rows < (int64_t)0x7fffffff, MOE_ERR_UNSUPPORTED);
  // bf16 on the tensor cores only: the gather is the tcgen05 kernel's A load
  if (!use_tc(cfg->act_dtype == MOE_BF16 ? kBF16 : kF32)) return MOE_ERR_UNSUPPORTED;
  MOE_PTR(w1); MOE_PTR(w2); MOE_OPT_PTR(pre_gu); MOE_OPT_PTR(offsets);
  if (n_rows > 0) { MOE_PTR(x); MOE_PTR(src_rows); MOE_PTR(h); MOE_PTR(out); }
  MOE_CTX(stream, c);
  c.act = glu_act_of(*cfg);
  if (n_rows == 0) return MOE_OK;
  int err = MOE_OK;
  MOE_LAUNCH(launch_tc_grouped_swiglu_fwd_gather(c, n_groups, n_rows, F, cfg->d, offsets, x,
                                                 x_rows, src_rows, w1, w2, pre_gu, h, out,
                                                 &err));
  return err;
}

int moe_unpermute_combine(const moe_cfg* cfg, const void* out_perm, const int32_t* row_of,
                          const float* w, const void* shared_out, const float* shared_gate,
                          void* y, moe_stream_t stream) {
  MOE_CHECK_CFG(cfg);
  if (cfg->T == 0) return MOE_OK;
  MOE_PTR(out_perm); MOE_PTR(row_of); MOE_PTR(w); MOE_PTR(y); MOE_OPT_PTR(shared_out);
  MOE_REQUIRE(shared_gate == nullptr || shared_out != nullptr, MOE_ERR_INVALID_ARG);
  MOE_REQUIRE(shared_gate == nullptr || (reinterpret_cast<uintptr_t>(shared_gate) & 3u) == 0,
              MOE_ERR_ALIGN);
  MOE_CTX(stream, c);
  MOE_LAUNCH(launch_combine(c, *cfg, out_perm, row_of, w, shared_out, shared_gate, y));
  return MOE_OK;
}

int moe_shared_gate(const moe_cfg* cfg, const void* x, const float* w_gate, float* gate,
                    moe_stream_t stream) {
  MOE_CHECK_CFG(cfg);
  if (cfg->T == 0) return MOE_OK;
  MOE_PTR(x); MOE_PTR(w_gate); MOE_PTR(gate);
  MOE_CTX(stream, c);
  MOE_LAUNCH(launch_shared_gate(c, *cfg, x, w_gate, gate));
  return MOE_OK;
}

int moe_shared_gate_bwd(const moe_cfg* cfg, const void* x, const float* gate, const void* dy,
                        const void* shared_out, void* dy_shared, float* d_gate_logit,
                        float* dw_gate, void* ws, size_t ws_bytes, moe_stream_t stream) {
  MOE_CHECK_CFG(cfg);
  MOE_PTR(dw_gate); MOE_PTR(ws);
  MOE_REQUIRE(ws_bytes >= shared_gate_bwd_ws(*cfg), MOE_ERR_WORKSPACE);
  if (cfg->T > 0) {
    MOE_PTR(x); MOE_PTR(gate); MOE_PTR(dy); MOE_PTR(shared_out); MOE_PTR(dy_shared);
    MOE_PTR(d_gate_logit);
  }
  MOE_CTX(stream, c);
  if (cfg->T == 0) {
    MOE_LAUNCH(cudaMemsetAsync(dw_gate, 0, (size_t)cfg->d * sizeof(float), c.stream));
    return MOE_OK;
  }
  MOE_LAUNCH(launch_shared_gate_bwd_tokens(c, *cfg, dy, shared_out, gate, dy_shared,
                                           d_gate_logit));
  // dw_gate = sum_t d_gate_logit[t] x[t]: the router's weight-gradient kernel
  // for a single expert, token slices summed in slice order
  moe_cfg one = *cfg;
  one.E = 1;
  const int S = route_bwd_splits(one);
  float* part = static_cast<float*>(ws);
  int used = S;
  MOE_LAUNCH(launch_router_dw_small(c, one, x, d_gate_logit, part, S, &used));
  MOE_LAUNCH(launch_reduce_partials(c, part, (int64_t)cfg->d, used, (int64_t)cfg->d, dw_gate,
                                    kF32, 0));
  return MOE_OK;
}

int moe_aux_loss(const moe_cfg* cfg, const float* logits, const int32_t* counts, float* aux,
                 void* ws, size_t ws_bytes, moe_stream_t stream) {
  MOE_CHECK_CFG(cfg);
  MOE_PTR(counts); MOE_PTR(ws);
  MOE_REQUIRE(aux != nullptr && (reinterpret_cast<uintptr_t>(aux) & 3u) == 0, MOE_ERR_INVALID_ARG);
  if (cfg->T > 0) MOE_PTR(logits);
  MOE_REQUIRE(ws_bytes >= aux_ws_bytes(*cfg), MOE_ERR_WORKSPACE);
  MOE_CTX(stream, c);
  MOE_LAUNCH(launch_aux_loss(c, *cfg, logits, counts, aux, ws));
  return MOE_OK;
}

int moe_unpermute_combine_bwd(const moe_cfg* cfg, const void* dy, const void* out_perm,
                              const int32_t* row_of, const float* w, void* d_out_perm, float* dw,
                              moe_stream_t stream) {
  MOE_CHECK_CFG(cfg);
  if (cfg->T == 0) return MOE_OK;
  MOE_PTR(dy); MOE_PTR(out_perm); MOE_PTR(row_of); MOE_PTR(w); MOE_PTR(d_out_perm); MOE_PTR(dw);
  MOE_CTX(stream, c);
  MOE_LAUNCH(launch_combine_bwd(c, *cfg, dy, out_perm, row_of, w, d_out_perm, dw));
  return MOE_OK;
}

int moe_grouped_swiglu_bwd(const moe_cfg* cfg, int32_t n_groups, int64_t n_rows, int32_t F,
                           const int32_t* offsets, const void* x_rows, const void* w1,
                           const void* w2, const void* pre_gu, const void* h, const void* d_out,
                           void* d_pre, void* dx_rows, void* dw1, void* dw2, void* ws,
                           size_t ws_bytes, moe_stream_t stream) {
  MOE_CHECK_CFG(cfg);
  MOE_REQUIRE(n_groups >= 1 && n_groups <= kMaxE && n_rows >= 0 && F > 0, MOE_ERR_INVALID_ARG);
  MOE_REQUIRE((F & 7) == 0, MOE_ERR_ALIGN);
  MOE_REQUIRE(offsets != nullptr || n_groups == 1, MOE_ERR_INVALID_ARG);
  MOE_REQUIRE(n_rows < (int64_t)0x7fffffff, MOE_ERR_UNSUPPORTED);
  MOE_PTR(w1); MOE_PTR(w2); MOE_PTR(dw1); MOE_PTR(dw2); MOE_OPT_PTR(offsets);
  if (n_rows > 0) {
    MOE_PTR(x_rows); MOE_PTR(pre_gu); MOE_PTR(h); MOE_PTR(d_out); MOE_PTR(d_pre); MOE_PTR(dx_rows);
    MOE_PTR(ws);
  }
  const size_t need_dh = round256((size_t)n_rows * F * sizeof(float));
  MOE_CTX(stream, c);
  c.act = glu_act_of(*cfg);
  const int dt = cfg->act_dtype == MOE_BF16 ? kBF16 : kF32;
  const int d = cfg->d;
  if (use_tc(dt)) {
    MOE_REQUIRE(ws_bytes >= round256(tc_grouped_ws_bytes(n_groups)), MOE_ERR_WORKSPACE);
    int err = MOE_OK;
    MOE_LAUNCH(launch_tc_grouped_swiglu_bwd(c, n_groups, n_rows, F, d, offsets, x_rows, w1, w2,
                                            pre_gu, h, d_out, d_pre, dx_rows, dw1, dw2, ws,
                                            ws_bytes, &err));
    return err;
  }
  MOE_REQUIRE(ws_bytes >= need_dh, MOE_ERR_WORKSPACE);
  float* dh = static_cast<float*>(ws);
  if (n_rows > 0) {
    SimtGemm a{};  // dh = d_out · W2_g      [rows, F]
    a.mode = kGroupM; a.M = (int)n_rows; a.N = F; a.K = d;
    a.dtA = dt; a.dtB = dt; a.dtC = kF32;
    a.A = d_out; a.a_sm = d; a.a_sk = 1;
    a.B = w2; a.b_sn = 1; a.b_sk = F; a.b_sg = (int64_t)d * F;
    a.C = dh; a.c_sm = F;
    a.offsets = offsets; a.n_groups = n_groups; a.alpha = 1.f;
    MOE_LAUNCH(launch_simt_gemm(c, a));
    MOE_LAUNCH(launch_swiglu_bwd_elem(c, dt, dh, pre_gu, d_pre, n_rows, F));
    SimtGemm b{};  // dx_rows = d_pre · W1_g [rows, d]
    b.mode = kGroupM; b.M = (int)n_rows; b.N = d; b.K = 2 * F;
    b.dtA = b.dtB = b.dtC = dt;
    b.A = d_pre; b.a_sm = 2 * F; b.a_sk = 1;
    b.B = w1; b.b_sn = 1; b.b_sk = d; b.b_sg = (int64_t)2 * F * d;
    b.C = dx_rows; b.c_sm = d;
    b.offsets = offsets; b.n_groups = n_groups; b.alpha = 1.f;
    MOE_LAUNCH(launch_simt_gemm(c, b));
  }
  SimtGemm w2g{};  // dW2_g = d_outᵀ · h   [d, F] per group, K = the group's rows
  w2g.mode = kGroupK; w2g.M = d; w2g.N = F; w2g.K = (int)n_rows;
  w2g.dtA = w2g.dtB = w2g.dtC = dt;
  w2g.A = d_out; w2g.a_sm = 1; w2g.a_sk = d;
  w2g.B = h; w2g.b_sn = 1; w2g.b_sk = F;
  w2g.C = dw2; w2g.c_sm = F; w2g.c_sg = (int64_t)d * F;
  w2g.offsets = offsets; w2g.n_groups = n_groups; w2g.alpha = 1.f;
  MOE_LAUNCH(launch_simt_gemm(c, w2g));
  SimtGemm w1g{};  // dW1_g = d_preᵀ · x_rows [2F, d] per group
  w1g.mode = kGroupK; w1g.M = 2 * F; w1g.N = d; w1g.K = (int)n_rows;
  w1g.dtA = w1g.dtB = w1g.dtC = dt;
  w1g.A = d_pre; w1g.a_sm = 1; w1g.a_sk = 2 * F;
  w1g.B = x_rows; w1g.b_sn = 1; w1g.b_sk = d;
  w1g.C = dw1; w1g.c_sm = d; w1g.c_sg = (int64_t)2 * F * d;
  w1g.offsets = offsets; w1g.n_groups = n_groups; w1g.alpha = 1.f;
  MOE_LAUNCH(launch_simt_gemm(c, w1g));
  return MOE_OK;
}

int moe_aux_loss_bwd(const moe_cfg* cfg, const float* logits, const int32_t* counts, float g_aux,
                     float* d_logits, int32_t accumulate, moe_stream_t stream) {
  MOE_CHECK_CFG(cfg);
  MOE_PTR(counts);
  if (cfg->T == 0) return MOE_OK;
  MOE_PTR(logits); MOE_PTR(d_logits);
  MOE_CTX(stream, c);
  MOE_LAUNCH(launch_aux_loss_bwd(c, *cfg, logits, counts, g_aux, d_logits, accumulate));
  return MOE_OK;
}

int moe_z_loss(const moe_cfg* cfg, const float* logits, float coeff, float* z, void* ws,
               size_t ws_bytes, moe_stream_t stream) {
  MOE_CHECK_CFG(cfg);
  MOE_PTR(z); MOE_PTR(ws);
  if (cfg->T > 0) { MOE_PTR(logits); }
  MOE_REQUIRE(ws_bytes >= z_loss_ws_bytes(*cfg), MOE_ERR_WORKSPACE);
  MOE_CTX(stream, c);
  MOE_LAUNCH(launch_z_loss(c, *cfg, logits, coeff, z, ws));
  return MOE_OK;
}

int moe_z_loss_bwd(const moe_cfg* cfg, const float* logits, float coeff, float g_z,
                   float* d_logits, int32_t accumulate, moe_stream_t stream) {
  MOE_CHECK_CFG(cfg);
  if (cfg->T == 0) return MOE_OK;
  MOE_PTR(logits); MOE_PTR(d_logits);
  MOE_CTX(stream, c);
  MOE_LAUNCH(launch_z_loss_bwd(c, *cfg, logits, coeff, g_z, d_logits, accumulate));
  return MOE_OK;
}

size_t moe_seq_aux_workspace_bytes(const moe_cfg* cfg, int64_t seq_len) {
  if (check_cfg(cfg) != MOE_OK) return 0;
  return seq_aux_ws_bytes(*cfg, seq_len);
}

int moe_seq_aux_loss(const moe_cfg* cfg, const float* logits, const int32_t* idx,
                     int64_t seq_len, int32_t seq_major, float coeff, float* out, void* ws,
                     size_t ws_bytes, moe_stream_t stream) {
  MOE_CHECK_CFG(cfg);
  MOE_REQUIRE(cfg->T > 0 && seq_len > 0 && cfg->T % seq_len == 0, MOE_ERR_INVALID_ARG);
  MOE_PTR(logits); MOE_PTR(idx); MOE_PTR(out); MOE_PTR(ws);
  MOE_REQUIRE(ws_bytes >= seq_aux_ws_bytes(*cfg, seq_len), MOE_ERR_WORKSPACE);
  MOE_CTX(stream, c);
  MOE_LAUNCH(launch_seq_aux_loss(c, *cfg, logits, idx, seq_len, seq_major != 0, coeff, out, ws));
  return MOE_OK;
}

int moe_seq_aux_loss_bwd(const moe_cfg* cfg, const float* logits, const int32_t* idx,
                         int64_t seq_len, int32_t seq_major, float coeff, float g,
                         float* d_logits, int32_t accumulate, void* ws, size_t ws_bytes,
                         moe_stream_t stream) {
  MOE_CHECK_CFG(cfg);
  MOE_REQUIRE(cfg->T > 0 && seq_len > 0 && cfg->T % seq_len == 0, MOE_ERR_INVALID_ARG);
  MOE_PTR(logits); MOE_PTR(idx); MOE_PTR(d_logits); MOE_PTR(ws);
  MOE_REQUIRE(ws_bytes >= seq_aux_ws_bytes(*cfg, seq_len), MOE_ERR_WORKSPACE);
  MOE_CTX(stream, c);
  MOE_LAUNCH(launch_seq_aux_loss_bwd(c, *cfg, logits, idx, seq_len, seq_major != 0, coeff, g,
                                     d_logits, accumulate, ws));
  return MOE_OK;
}

int moe_tokens_per_expert_accumulate(const moe_cfg* cfg, const int32_t* counts,
                                     int64_t* tokens_per_expert, moe_stream_t stream) {
  MOE_CHECK_CFG(cfg);
  MOE_PTR(counts); MOE_PTR(tokens_per_expert);
  MOE_CTX(stream, c);
  MOE_LAUNCH(launch_tokens_accumulate(c, *cfg, counts, tokens_per_expert));
  return MOE_OK;
}

int moe_expert_bias_update(const moe_cfg* cfg, const int64_t* tokens_per_expert,
                           float* expert_bias, float rate, moe_stream_t stream) {
  MOE_CHECK_CFG(cfg);
  MOE_PTR(tokens_per_expert); MOE_PTR(expert_bias);
  MOE_CTX(stream, c);
  MOE_LAUNCH(launch_expert_bias_update(c, *cfg, tokens_per_expert, expert_bias, rate));
  return MOE_OK;
}

int moe_max_vio(const moe_cfg* cfg, const int64_t* tokens_per_expert, float* max_vio,
                moe_stream_t stream) {
  MOE_CHECK_CFG(cfg);
  MOE_PTR(tokens_per_expert); MOE_PTR(max_vio);
  MOE_CTX(stream, c);
  MOE_LAUNCH(launch_max_vio(c, *cfg, tokens_per_expert, max_vio));
  return MOE_OK;
}

int moe_gate_logits(const moe_cfg* cfg, const void* x, const float* w_router,
                    const float* logit_bias, float* logits, void* ws, size_t ws_bytes,
                    moe_stream_t stream) {
  MOE_CHECK_CFG(cfg);
  if (cfg->T == 0) return MOE_OK;
  MOE_PTR(x); MOE_PTR(w_router); MOE_PTR(logits);
  MOE_REQUIRE(logit_bias == nullptr || (reinterpret_cast<uintptr_t>(logit_bias) & 3u) == 0, MOE_ERR_ALIGN);
  const size_t need = router_ws_bytes(*cfg);
  MOE_REQUIRE(ws_bytes >= need, MOE_ERR_WORKSPACE);
  if (need > 0) { MOE_PTR(ws); }
  MOE_CTX(stream, c);
  MOE_LAUNCH(launch_router_logits(c, *cfg, x, w_router, logit_bias, logits,
                                  need > 0 ? ws : nullptr));
  return MOE_OK;
}

int moe_quantile_route(const moe_cfg* cfg, const float* logits, const float* beta,
                       int32_t* idx, float* w, float* alpha, float* beta_local,
                       moe_stream_t stream) {
  MOE_CHECK_CFG(cfg);
  MOE_REQUIRE(cfg->score_fn != MOE_SCORE_SOFTMAX_PRE, MOE_ERR_UNSUPPORTED);
  MOE_REQUIRE(cfg->k < cfg->E, MOE_ERR_INVALID_ARG);
  if (beta_local != nullptr) {
    MOE_REQUIRE(cfg->T > 0 && (cfg->T * (int64_t)cfg->k) % cfg->E == 0, MOE_ERR_INVALID_ARG);
    MOE_PTR(beta_local);
  }
  MOE_PTR(beta); MOE_PTR(alpha);
  if (cfg->T > 0) { MOE_PTR(logits); MOE_PTR(idx); MOE_PTR(w); }
  MOE_CTX(stream, c);
  MOE_LAUNCH(launch_router_topk_q(c, *cfg, logits, nullptr, beta, alpha, idx, w));
  if (beta_local != nullptr) MOE_LAUNCH(launch_quantile_solve(c, *cfg, logits, alpha, beta_local));
  return MOE_OK;
}

int moe_quantile_accumulate(const moe_cfg* cfg, const float* beta_local, float* accum,
                            int32_t* count, moe_stream_t stream) {
  MOE_CHECK_CFG(cfg);
  MOE_PTR(beta_local); MOE_PTR(accum); MOE_PTR(count);
  MOE_CTX(stream, c);
  MOE_LAUNCH(launch_quantile_accumulate(c, *cfg, beta_local, accum, count));
  return MOE_OK;
}

int moe_quantile_beta_update(const moe_cfg* cfg, float* beta, float* accum, int32_t* count,
                             float ema, moe_stream_t stream) {
  MOE_CHECK_CFG(cfg);
  MOE_REQUIRE(ema >= 0.f && ema <= 1.f, MOE_ERR_INVALID_ARG);
  MOE_PTR(beta); MOE_PTR(accum); MOE_PTR(count);
  MOE_CTX(stream, c);
  MOE_LAUNCH(launch_quantile_beta_update(c, *cfg, beta, accum, count, ema));
  return MOE_OK;
}

int moe_route_topk_bwd(const moe_cfg* cfg, const void* x, const float* w_router,
                       const float* logits, const int32_t* idx, const float* dw, float* d_logits,
                       int32_t accumulate, float* dx_router, float* dw_router, void* ws,
                       size_t ws_bytes, moe_stream_t stream) {
  MOE_CHECK_CFG(cfg);
  MOE_PTR(w_router); MOE_PTR(dw_router); MOE_PTR(ws);
  MOE_REQUIRE(ws_bytes >= route_bwd_ws(*cfg), MOE_ERR_WORKSPACE);
  if (cfg->T > 0) {
    MOE_PTR(x); MOE_PTR(logits); MOE_PTR(idx); MOE_PTR(dw); MOE_PTR(d_logits);
    MOE_OPT_PTR(dx_router);
  }
  // dx_router NULL: the caller has moe_permute_bwd form d_logits · W_r
  if (dx_router == nullptr && !permute_bwd_forms_router_dx(*cfg)) return MOE_ERR_INVALID_ARG;
  MOE_CTX(stream, c);
  const int dtx = cfg->act_dtype == MOE_BF16 ? kBF16 : kF32;
  const int T = (int)cfg->T, E = cfg->E, d = cfg->d;
  MOE_LAUNCH(launch_router_scores_bwd(c, *cfg, logits, idx, dw, d_logits, accumulate));
  if (T > 0 && router_bwd_tc_eligible(*cfg)) {
    MOE_LAUNCH(launch_router_bwd_tc(c, *cfg, x, w_router, d_logits, dx_router, dw_router, ws));
    return MOE_OK;
  }
  if (T > 0 && dx_router == nullptr) {
    // formed later by moe_permute_bwd
  } else if (T > 0 && E <= 16) {
    MOE_LAUNCH(launch_router_dx_small(c, *cfg, d_logits, w_router, dx_router));
  } else if (T > 0) {
    SimtGemm a{};  // dx_router = d_logits · W_r   [T, d], K = E
    a.mode = kGroupNone; a.M = T; a.N = d; a.K = E;
    a.dtA = kF32; a.dtB = kF32; a.dtC = kF32;
    a.A = d_logits; a.a_sm = E; a.a_sk = 1;
    a.B = w_router; a.b_sn = 1; a.b_sk = d;
    a.C = dx_router; a.c_sm = d;
    a.n_groups = 1; a.alpha = 1.f; a.split_k = 1;
    MOE_LAUNCH(launch_simt_gemm(c, a));
  }
  const int S = route_bwd_splits(*cfg);
  float* part = static_cast<float*>(ws);
  // dW_r = d_logitsᵀ · x [E, d], K = T split S ways. Computed as its transpose
  // (M = d, N = E) so that the 128-row tiles run along d, written back as [E, d].
  SimtGemm b{};
  b.mode = kGroupNone; b.M = d; b.N = E; b.K = T;
  b.dtA = dtx; b.dtB = kF32; b.dtC = kF32;
  b.A = x; b.a_sm = 1; b.a_sk = d;
  b.B = d_logits; b.b_sn = 1; b.b_sk = E;
  b.C = part; b.c_sm = 1; b.c_sn = d; b.c_sg = (int64_t)E * d;
  b.n_groups = 1; b.alpha = 1.f; b.split_k = S;
  if (T > 0) {
    int used = S;
    if (E <= 16) {
      MOE_LAUNCH(launch_router_dw_small(c, *cfg, x, d_logits, part, S, &used));
    } else {
      MOE_LAUNCH(launch_simt_gemm(c, b));
    }
    MOE_LAUNCH(launch_reduce_partials(c, part, (int64_t)E * d, used, (int64_t)E * d, dw_router,
                                      kF32, 0));
  } else {
    MOE_LAUNCH(cudaMemsetAsync(dw_router, 0, (size_t)E * d * sizeof(float), c.stream));
  }
  return MOE_OK;
}

int moe_permute_bwd(const moe_cfg* cfg, const void* dx_perm, const int32_t* row_of,
                    const float* dx_router, const void* dx_shared, const float* d_gate_logit,
                    const float* w_gate, const float* d_logits, const float* w_router, void* dx,
                    moe_stream_t stream) {
  MOE_CHECK_CFG(cfg);
  if (cfg->T == 0) return MOE_OK;  // (empty buffers may come as NULL)
  MOE_REQUIRE((d_gate_logit == nullptr) == (w_gate == nullptr), MOE_ERR_INVALID_ARG);
  MOE_REQUIRE((d_logits == nullptr) == (w_router == nullptr), MOE_ERR_INVALID_ARG);
  MOE_REQUIRE(d_logits == nullptr || dx_router == nullptr, MOE_ERR_INVALID_ARG);
  if (d_logits != nullptr && !permute_bwd_forms_router_dx(*cfg)) return MOE_ERR_UNSUPPORTED;
  MOE_PTR(dx_perm); MOE_PTR(row_of); MOE_PTR(dx); MOE_OPT_PTR(dx_router); MOE_OPT_PTR(dx_shared);
  MOE_OPT_PTR(d_gate_logit); MOE_OPT_PTR(w_gate); MOE_OPT_PTR(d_logits); MOE_OPT_PTR(w_router);
  MOE_CTX(stream, c);
  MOE_LAUNCH(launch_permute_bwd(c, *cfg, dx_perm, row_of, dx_router, dx_shared, d_gate_logit,
                                w_gate, d_logits, w_router, dx));
  return MOE_OK;
}

int moe_router_dx_in_permute_bwd(const moe_cfg* cfg) {
  MOE_CHECK_CFG(cfg);
  return permute_bwd_forms_router_dx(*cfg) ? 1 : 0;
}

// ---- dispatch with a fixed device scratch array (no allocation by anyone)
}  // extern "C"

namespace moe {
// The scratch of moe_permute_noalloc: per-block expert counts, then bases.
// In host code this name is only a stand-in; its device address comes from
// cudaGetSymbolAddress, looked up once per device with that device current.
static __device__ __align__(256) int32_t g_noalloc_scratch[MOE_PERMUTE_NOALLOC_SCRATCH_BYTES / 4];
static std::mutex g_noalloc_mu;
static int32_t* g_noalloc_ptr[kMaxDevices];
}  // namespace moe

extern "C" {

int moe_permute_noalloc(const moe_cfg* cfg, const void* x, const int32_t* idx, int32_t* counts,
                        int32_t* offsets, int32_t* row_of, int32_t* src_tok, void* x_perm,
                        moe_stream_t stream) {
  MOE_CHECK_CFG(cfg);
  MOE_PTR(counts); MOE_PTR(offsets);
  if (cfg->T > 0) {
    MOE_PTR(x); MOE_PTR(idx); MOE_PTR(row_of); MOE_PTR(src_tok); MOE_PTR(x_perm);
  }
  if (permute_ws_bytes(*cfg) > sizeof(g_noalloc_scratch)) return MOE_ERR_UNSUPPORTED;
  MOE_CTX(stream, c);
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) {
    cudaGetLastError();
    return MOE_ERR_NO_DEVICE;
  }
  int32_t* scratch = nullptr;
  {
    std::lock_guard<std::mutex> lk(g_noalloc_mu);
    if (g_noalloc_ptr[dev] == nullptr) {
      void* p = nullptr;
      if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || p == nullptr) {
        cudaGetLastError();
        return MOE_ERR_CUDA;
      }
      g_noalloc_ptr[dev] = static_cast<int32_t*>(p);
    }
    scratch = g_noalloc_ptr[dev];
  }
  MOE_LAUNCH(launch_permute(c, *cfg, x, idx, counts, offsets, row_of, src_tok, x_perm, scratch));
  return MOE_OK;
}

int moe_selftest_wait_timeout(moe_stream_t stream) {
  MOE_CTX(stream, c);
  MOE_LAUNCH(launch_wait_selftest(c));
  return MOE_OK;
}

}  // extern "C"

namespace moe {

// Waits for status[2], which nothing sets, until the timeout; records
// MOE_ERR_TIMEOUT (detail 1) and returns.
__global__ void wait_selftest_kernel(int* status, uint64_t timeout_ns) {
  if (threadIdx.x != 0) return;
  volatile int* flag = status + 2;
  const uint64_t t0 = global_timer_ns();
  while (*flag == 0) {
    if (global_timer_ns() - t0 > timeout_ns) {
      record_error(status, MOE_ERR_TIMEOUT, 1);
      return;
    }
    __nanosleep(1000);
  }
}

cudaError_t launch_wait_selftest(const Ctx& c) {
  wait_selftest_kernel<<<1, 32, 0, c.stream>>>(c.status, c.timeout_ns);
  note_launches(1);
  return cudaGetLastError();
}

}  // namespace moe
