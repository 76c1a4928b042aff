// Launchers shared between the kernel files and the C-ABI file (C++ linkage).
#pragma once

#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include "moe.h"

namespace moe {

// score functions that take the aux-loss-free selection bias (Megatron refuses
// it with softmax, before or after the top-k)
inline bool score_takes_bias(int score_fn) {
  return score_fn == MOE_SCORE_SIGMOID || score_fn == MOE_SCORE_SQRT_SOFTPLUS;
}

// expert activation (moe_cfg's act_* fields); fn = MOE_ACT_*
struct GluAct {
  int fn;
  float clamp, gate_scale, linear_scale, offset;
};
inline GluAct glu_act_of(const moe_cfg& cfg) {
  return GluAct{cfg.act_fn, cfg.act_clamp, cfg.act_gate_scale, cfg.act_linear_scale,
                cfg.glu_linear_offset};
}
__host__ __device__ inline bool glu_is_plain(const GluAct& a) {
  return a.fn == MOE_ACT_SWIGLU && a.offset == 0.f;
}

struct Ctx {
  cudaStream_t stream;
  int* status;          // device status word of the current device
  uint64_t timeout_ns;  // bound of every spin-wait
  int sm_count;
  GluAct act;           // the call's expert activation (grouped SwiGLU calls)
};

// ---- router (router.cu; tensor-core gate GEMM in router_tc.cu)
// ws: the router workspace (router_ws_bytes) or NULL when that size is 0
cudaError_t launch_router_logits(const Ctx& c, const moe_cfg& cfg, const void* x,
                                 const float* w_router, const float* logit_bias,
                                 float* logits, void* ws);
size_t router_ws_bytes(const moe_cfg& cfg);
bool router_tc_eligible(const moe_cfg& cfg);
int router_set_impl(int impl);    // 0 tensor cores where eligible, 1 CUDA cores
bool router_tensor_cores_enabled();
// router backward on the tensor cores (router_bwd_tc.cu): dx_router and dW_r
bool router_bwd_tc_shape(const moe_cfg& cfg);     // a shape the kernels take
bool router_bwd_tc_eligible(const moe_cfg& cfg);  // shape, setting and driver allow it
size_t router_bwd_tc_ws_bytes(const moe_cfg& cfg);
cudaError_t launch_router_bwd_tc(const Ctx& c, const moe_cfg& cfg, const void* x,
                                 const float* w_router, const float* d_logits, float* dx_router,
                                 float* dw_router, void* ws);
int router_set_fold(int fold_k);  // K elements per compensated window (multiple of 16)
cudaError_t launch_router_logits_tc(const Ctx& c, const moe_cfg& cfg, const void* x_bf16,
                                    const float* w_router, const float* logit_bias,
                                    float* logits, void* ws);
cudaError_t launch_router_topk(const Ctx& c, const moe_cfg& cfg, const float* logits,
                               const float* sel_bias, int32_t* idx, float* w);
// top-k with a quantile bias: key = score - beta, k + 1 ranked, alpha[t] =
// the (k+1)-th key (beta, alpha NULL: plain top-k)
cudaError_t launch_router_topk_q(const Ctx& c, const moe_cfg& cfg, const float* logits,
                                 const float* sel_bias, const float* beta, float* alpha,
                                 int32_t* idx, float* w);
// quantile balancing (quantile.cu)
cudaError_t launch_quantile_solve(const Ctx& c, const moe_cfg& cfg, const float* logits,
                                  const float* alpha, float* beta_local);
cudaError_t launch_quantile_accumulate(const Ctx& c, const moe_cfg& cfg, const float* beta_local,
                                       float* accum, int32_t* count);
cudaError_t launch_quantile_beta_update(const Ctx& c, const moe_cfg& cfg, float* beta,
                                        float* accum, int32_t* count, float ema);
// dW_r partials [used][E][d] for E <= 16, used <= splits token slices (sum
// them in slice order)
cudaError_t launch_router_dw_small(const Ctx& c, const moe_cfg& cfg, const void* x,
                                   const float* d_logits, float* part, int splits, int* used);
// dx_router = d_logits · W_r for E <= 16 (fp32, experts summed in order)
cudaError_t launch_router_dx_small(const Ctx& c, const moe_cfg& cfg, const float* d_logits,
                                   const float* w_router, float* dx_router);
cudaError_t launch_router_near_ties(const Ctx& c, const moe_cfg& cfg, const float* logits,
                                    const float* sel_bias, float band, int32_t* count);
cudaError_t launch_router_scores_bwd(const Ctx& c, const moe_cfg& cfg, const float* logits,
                                     const int32_t* idx, const float* dw, float* d_logits,
                                     int accumulate);

// ---- router z-loss and sequence-wise aux loss (aux_loss.cu)
size_t z_loss_ws_bytes(const moe_cfg& cfg);
cudaError_t launch_z_loss(const Ctx& c, const moe_cfg& cfg, const float* logits, float coeff,
                          float* z, void* ws);
cudaError_t launch_z_loss_bwd(const Ctx& c, const moe_cfg& cfg, const float* logits, float coeff,
                              float g_z, float* d_logits, int accumulate);
size_t seq_aux_ws_bytes(const moe_cfg& cfg, int64_t seq_len);  // 0: seq_len does not divide T
cudaError_t launch_seq_aux_loss(const Ctx& c, const moe_cfg& cfg, const float* logits,
                                const int32_t* idx, int64_t seq_len, int seq_major, float coeff,
                                float* out, void* ws);
cudaError_t launch_seq_aux_loss_bwd(const Ctx& c, const moe_cfg& cfg, const float* logits,
                                    const int32_t* idx, int64_t seq_len, int seq_major,
                                    float coeff, float g, float* d_logits, int accumulate,
                                    void* ws);

// ---- load-balance bookkeeping (balance.cu)
cudaError_t launch_tokens_accumulate(const Ctx& c, const moe_cfg& cfg, const int32_t* counts,
                                     int64_t* tokens_per_expert);
cudaError_t launch_expert_bias_update(const Ctx& c, const moe_cfg& cfg,
                                      const int64_t* tokens_per_expert, float* expert_bias,
                                      float rate);
cudaError_t launch_max_vio(const Ctx& c, const moe_cfg& cfg, const int64_t* tokens_per_expert,
                           float* out);

// ---- dispatch (dispatch.cu)
size_t permute_ws_bytes(const moe_cfg& cfg);
cudaError_t launch_permute(const Ctx& c, const moe_cfg& cfg, const void* x, const int32_t* idx,
                           int32_t* counts, int32_t* offsets, int32_t* row_of,
                           int32_t* src_tok, void* x_perm, void* ws);
cudaError_t launch_permute_bwd(const Ctx& c, const moe_cfg& cfg, const void* dx_perm,
                               const int32_t* row_of, const float* dx_router,
                               const void* dx_shared, const float* d_gate_logit,
                               const float* w_gate, const float* d_logits,
                               const float* w_router, void* dx);
// whether moe_permute_bwd forms the router's input gradient d_logits · W_r
// itself (few experts) rather than reading it as dx_router
bool permute_bwd_forms_router_dx(const moe_cfg& cfg);

// ---- combine (combine.cu)
cudaError_t launch_combine(const Ctx& c, const moe_cfg& cfg, const void* out_perm,
                           const int32_t* row_of, const float* w, const void* shared_out,
                           const float* shared_gate, void* y);
// the shared expert's sigmoid gate (shared_gate.cu)
cudaError_t launch_shared_gate(const Ctx& c, const moe_cfg& cfg, const void* x,
                               const float* w_gate, float* gate);
cudaError_t launch_shared_gate_bwd_tokens(const Ctx& c, const moe_cfg& cfg, const void* dy,
                                          const void* shared_out, const float* gate,
                                          void* dy_shared, float* d_gate_logit);
cudaError_t launch_combine_bwd(const Ctx& c, const moe_cfg& cfg, const void* dy,
                               const void* out_perm, const int32_t* row_of, const float* w,
                               void* d_out_perm, float* dw);

// ---- aux loss (aux_loss.cu)
size_t aux_ws_bytes(const moe_cfg& cfg);
cudaError_t launch_aux_loss(const Ctx& c, const moe_cfg& cfg, const float* logits,
                            const int32_t* counts, float* aux, void* ws);
cudaError_t launch_aux_loss_bwd(const Ctx& c, const moe_cfg& cfg, const float* logits,
                                const int32_t* counts, float g_aux, float* d_logits,
                                int accumulate);

// ---- generic fp32-accumulating SIMT GEMM (simt_gemm.cu)
// C(m, n) = alpha * sum_k A(m, k) * B(n, k)  (+ C(m, n) when accumulate)
// A(m, k) = A[m*a_sm + k*a_sk], B(n, k) = B[n*b_sn + k*b_sk], C(m, n) = C[m*c_sm + n*c_sn].
enum SimtGrouping { kGroupNone = 0, kGroupM = 1, kGroupK = 2 };
enum SimtDtype { kF32 = 0, kBF16 = 1 };
struct SimtGemm {
  int mode;                // SimtGrouping
  int M, N, K;             // kGroupM: M = total rows; kGroupK: K = total rows
  int dtA, dtB, dtC;       // SimtDtype
  const void* A; int64_t a_sm, a_sk, a_sg;
  const void* B; int64_t b_sn, b_sk, b_sg;
  void* C; int64_t c_sm, c_sg;
  int64_t c_sn;            // C(m, n) = C[m*c_sm + n*c_sn]; 0 means 1
  const int32_t* offsets;  // [n_groups + 1] device (grouped modes), NULL = one group
  int n_groups;
  float alpha;
  int accumulate;
  int split_k;             // kGroupNone only: >1 writes partials C + z*c_sg, then reduce
};
cudaError_t launch_simt_gemm(const Ctx& c, const SimtGemm& g);
// out[i] = sum_z part[z*stride + i] (fixed order), i < n; dtype of out: dt_out
cudaError_t launch_reduce_partials(const Ctx& c, const float* part, int64_t stride, int nz,
                                   int64_t n, void* out, int dt_out, int accumulate);

// ---- SwiGLU elementwise (simt_gemm.cu)
cudaError_t launch_swiglu_fwd_elem(const Ctx& c, int dt, const void* pre_gu, void* h,
                                   int64_t rows, int F);
cudaError_t launch_swiglu_bwd_elem(const Ctx& c, int dt, const float* dh, const void* pre_gu,
                                   void* d_pre, int64_t rows, int F);

// ---- tcgen05 grouped GEMM (grouped_gemm_tc.cu)
struct TcGroupedArgs;
bool tc_available();
cudaError_t launch_tc_grouped_swiglu_fwd(const Ctx& c, int n_groups, int64_t n_rows, int F,
                                         int d, const int32_t* offsets, const void* x_rows,
                                         const void* w1, const void* w2, void* pre_gu,
                                         void* h, void* out, void* ws, int* err);
// fc1 with its A rows gathered from x through src_rows (x_rows rows in x),
// then fc2; single CTAs for fc1
cudaError_t launch_tc_grouped_swiglu_fwd_gather(const Ctx& c, int G, int64_t n_rows, int F, int d,
                                                const int32_t* offsets, const void* x,
                                                int64_t x_rows, const int32_t* src_rows,
                                                const void* w1, const void* w2, void* pre_gu,
                                                void* h, void* out, int* err);
cudaError_t launch_tc_grouped_swiglu_bwd(const Ctx& c, int n_groups, int64_t n_rows, int F,
                                         int d, const int32_t* offsets, const void* x_rows,
                                         const void* w1, const void* w2, const void* pre_gu,
                                         const void* h, const void* d_out, void* d_pre,
                                         void* dx_rows, void* dw1, void* dw2, void* ws,
                                         size_t ws_bytes, int* err);
size_t tc_grouped_ws_bytes(int n_groups);
// workspace the grouped backward uses, when present, for the weight
// gradients' per-expert tail tensor maps (two per group)
size_t tc_tail_maps_bytes(int n_groups);
// kernel kinds of the grouped GEMM, for per-kernel timing
enum TcKind { kFc1Fwd = 0, kFc2Fwd, kFc2Dgrad, kFc1Dgrad, kFc2Wgrad, kFc1Wgrad, kTcKinds };
int tc_timing_enable(int on);
int tc_set_mode(int mode);  // 0 auto, 1 single-CTA only, 2 CTA pairs always
int tc_timing_read(float* ms_total, int32_t* launches);

// ---- misc
cudaError_t launch_wait_selftest(const Ctx& c);
// host-side count of kernels this library has launched (for the bench's claim)
void note_launches(int n);
uint64_t launches_so_far();

}  // namespace moe
