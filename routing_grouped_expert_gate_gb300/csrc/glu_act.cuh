// Expert activations on fc1's [gate | linear] halves and their derivatives.
//
// The Ultimate MoE Training Handbook §3.4 "Experts", part "Activation" (the
// glu() of Megatron's MLP and the SiTU-GLU of Kimi K3):
//   SwiGLU        h = silu(g) * (u + offset)
//   SwiGLU clamp  h = silu(min(g, c)) * clamp(u, -c, c); a clipped input passes
//                 no gradient (the clip's derivative is 1 on [-c, c], ends
//                 included, 0 outside)
//   SiTU-GLU      h = s tanh(g / s) sigmoid(g) * (lin(u) + offset),
//                 lin(u) = s_l tanh(u / s_l) when s_l > 0, else u
#pragma once
#include "common.cuh"
#include "internal.h"

namespace moe {

__device__ __forceinline__ float glu_sig(float z) { return 1.f / (1.f + __expf(-z)); }

__device__ __forceinline__ float glu_fwd(float g, float u, const GluAct& a) {
  if (a.fn == MOE_ACT_SWIGLU_CLAMP) {
    const float gc = fminf(g, a.clamp);
    const float uc = fminf(fmaxf(u, -a.clamp), a.clamp);
    return gc * glu_sig(gc) * uc;
  }
  if (a.fn == MOE_ACT_SITU_GLU) {
    const float s = a.gate_scale;
    const float gate = s * tanhf(g / s) * glu_sig(g);
    const float lin = a.linear_scale > 0.f ? a.linear_scale * tanhf(u / a.linear_scale) : u;
    return gate * (lin + a.offset);
  }
  return g * glu_sig(g) * (u + a.offset);
}

__device__ __forceinline__ void glu_bwd(float g, float u, float dh, const GluAct& a, float& dg,
                                        float& du) {
  if (a.fn == MOE_ACT_SWIGLU_CLAMP) {
    const float c = a.clamp;
    const float gc = fminf(g, c), uc = fminf(fmaxf(u, -c), c);
    const float sg = glu_sig(gc);
    dg = (g <= c) ? dh * uc * sg * (1.f + gc * (1.f - sg)) : 0.f;
    du = (u >= -c && u <= c) ? dh * gc * sg : 0.f;
    return;
  }
  if (a.fn == MOE_ACT_SITU_GLU) {
    const float s = a.gate_scale;
    const float th = tanhf(g / s), sg = glu_sig(g);
    const float gate = s * th * sg;
    const float dgate = (1.f - th * th) * sg + s * th * sg * (1.f - sg);
    float lin = u, dlin = 1.f;
    if (a.linear_scale > 0.f) {
      const float tl = tanhf(u / a.linear_scale);
      lin = a.linear_scale * tl;
      dlin = 1.f - tl * tl;
    }
    dg = dh * (lin + a.offset) * dgate;
    du = dh * gate * dlin;
    return;
  }
  const float sg = glu_sig(g);
  dg = dh * (u + a.offset) * sg * (1.f + g * (1.f - sg));
  du = dh * g * sg;
}

}  // namespace moe
