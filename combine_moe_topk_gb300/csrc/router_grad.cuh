// router_grad.cuh -- the top-k gate backward of one token, for one warp:
// the router logits' gradient from the gradients of the token's k gates.
//
// DeepSpeed #8213 "Add an opt-in DeepEP transport for the AutoEP expert
// all-to-all", review thread: the gradient of the routing weights must reach
// the router.  With g = the gates of the selected experts:
//   renorm (g = softmax over the k selected logits):
//     dlogit_x = g_x (dg_x - c) for a selected x, 0 otherwise;
//   no renorm (g = the full softmax probability p_x):
//     dlogit_x = p_x (dg_x - c) for every x (dg_x = 0 when x is not selected);
//   c = sum_j g_j dg_j.
// Used by the gate backward kernel and, fused, by the combine backward, so
// both give the same bits: lanes 0..k-1 hold (expert, gate, gate gradient)
// of the token's routes; c is a butterfly over the warp; lane l writes the
// experts l, l + 32, ... (EPL of them; entries past e are skipped, so a
// larger EPL than e needs computes the same values).
#pragma once

#include <math.h>

#include "common.cuh"

namespace moe {

template <int EPL>
__device__ __forceinline__ void router_grad_token(int t, int lane, int k, int e, int renorm, int ij,
                                                  float gj, float dgj,
                                                  const float* __restrict__ logits,
                                                  float* __restrict__ dlogits) {
  float c = __fmul_rn(gj, dgj);  // lanes past k hold gj = dgj = 0
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) c += __shfl_xor_sync(0xffffffffu, c, off);
  // this lane's experts: their gate gradient (0 if not selected) and factor
  float dg[EPL], fac[EPL];
#pragma unroll
  for (int i = 0; i < EPL; ++i) {
    dg[i] = 0.f;
    fac[i] = 0.f;
  }
  for (int j = 0; j < k; ++j) {
    const int x = __shfl_sync(0xffffffffu, ij, j);
    const float g = __shfl_sync(0xffffffffu, gj, j);
    const float d = __shfl_sync(0xffffffffu, dgj, j);
#pragma unroll
    for (int i = 0; i < EPL; ++i)
      if (lane + 32 * i == x) {
        dg[i] = d;
        fac[i] = g;
      }
  }
  if (!renorm) {
    const float* l = logits + (size_t)t * e;
    float v[EPL];
    float mx = -INFINITY;
#pragma unroll
    for (int i = 0; i < EPL; ++i) {
      const int x = lane + 32 * i;
      v[i] = x < e ? __ldg(l + x) : -INFINITY;
      mx = fmaxf(mx, v[i]);
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, off));
    float z = 0.f;
#pragma unroll
    for (int i = 0; i < EPL; ++i)
      if (lane + 32 * i < e) z += expf(v[i] - mx);
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) z += __shfl_xor_sync(0xffffffffu, z, off);
#pragma unroll
    for (int i = 0; i < EPL; ++i) fac[i] = expf(v[i] - mx) / z;  // p_x for every expert
  }
  float* out = dlogits + (size_t)t * e;
#pragma unroll
  for (int i = 0; i < EPL; ++i) {
    const int x = lane + 32 * i;
    // an expert outside the top-k gets exactly 0 under renormalisation
    if (x < e) out[x] = fac[i] == 0.f ? 0.f : __fmul_rn(fac[i], __fsub_rn(dg[i], c));
  }
}

}  // namespace moe
