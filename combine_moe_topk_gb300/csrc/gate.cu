// gate.cu -- top-k softmax gating and its backward, one warp per token.
//
// DeepSpeed #8195 "MoE dispatch: fix silent Tutel + TP corruption, speed up
// native and Tutel paths", change 1: the gate hands out per-route expert
// index and weight directly (no dense [s, e] mask per route), as contiguous
// int32 routes.  Automodel #3684 "perf(moe): reuse the DeepEP dispatch
// layout on activation-checkpoint recompute": a recompute must route
// exactly as the forward did, so selection is a pure comparison on the
// logits (no exp rounding can change it) with a fixed tie-break.
//
// The selection of one token by one warp is topk_gate_kernel's loop body,
// topk_token (gate_core.cuh); this file adds the launch shape (a warp per
// token, the next token's logits loaded one token ahead) and the backward.
#include <math.h>

#include "common.cuh"
#include "gate_core.cuh"
#include "internal.h"
#include "router_grad.cuh"

namespace moe {

namespace {

template <int EPL>
__global__ void __launch_bounds__(256) topk_gate_kernel(const float* __restrict__ logits, int s,
                                                        int e, int k, int renorm,
                                                        int32_t* __restrict__ idx,
                                                        float* __restrict__ gate,
                                                        int32_t* status) {
  const int lane = threadIdx.x & 31;
  const int warps = (gridDim.x * blockDim.x) >> 5;
  grid_dependency_wait();
  pdl_trigger_early();
  // this lane's logits of the warp's next token are loaded one token ahead,
  // so their latency overlaps the current token's selection
  int t = (blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  float nxt[EPL];
#pragma unroll
  for (int i = 0; i < EPL; ++i) {
    const int j = lane + 32 * i;
    nxt[i] = (t < s && j < e) ? __ldg(logits + (size_t)t * e + j) : 0.0f;
  }
  for (; t < s; t += warps) {
    float cur[EPL];
#pragma unroll
    for (int i = 0; i < EPL; ++i) cur[i] = nxt[i];
    const int tn = t + warps;
#pragma unroll
    for (int i = 0; i < EPL; ++i) {
      const int j = lane + 32 * i;
      nxt[i] = (tn < s && j < e) ? __ldg(logits + (size_t)tn * e + j) : 0.0f;
    }
    int sel_id;
    float g;
    if (topk_token<EPL>(cur, lane, e, k, renorm, &sel_id, &g) && lane == 0) raise_status(status, MOE_DEV_NONFINITE);
    if (lane < k) {
      idx[(size_t)t * k + lane] = sel_id;
      gate[(size_t)t * k + lane] = g;
    }
  }
  pdl_trigger_late();
}

// Gate backward, one warp per token: lanes 0..k-1 hold (expert, gate,
// dgate) of the selected routes; router_grad_token does the rest.
template <int EPL>
__global__ void __launch_bounds__(256) topk_gate_bwd_kernel(
    const float* __restrict__ logits, const int32_t* __restrict__ idx,
    const float* __restrict__ gate, const float* __restrict__ dgate, int s, int e, int k,
    int renorm, float* __restrict__ dlogits) {
  const int lane = threadIdx.x & 31;
  const int warps = (gridDim.x * blockDim.x) >> 5;
  grid_dependency_wait();
  pdl_trigger_early();
  // the route data of the warp's next token is loaded one token ahead
  int t = (blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  int n_ij = -1;
  float n_gj = 0.f, n_dgj = 0.f;
  if (t < s && lane < k) {
    n_ij = __ldg(idx + (size_t)t * k + lane);
    n_gj = __ldg(gate + (size_t)t * k + lane);
    n_dgj = __ldg(dgate + (size_t)t * k + lane);
  }
  for (; t < s; t += warps) {
    const int ij = n_ij;
    const float gj = n_gj, dgj = n_dgj;
    const int tn = t + warps;
    if (tn < s && lane < k) {
      n_ij = __ldg(idx + (size_t)tn * k + lane);
      n_gj = __ldg(gate + (size_t)tn * k + lane);
      n_dgj = __ldg(dgate + (size_t)tn * k + lane);
    }
    router_grad_token<EPL>(t, lane, k, e, renorm, ij, gj, dgj, logits, dlogits);
  }
  pdl_trigger_late();
}

template <int EPL>
cudaError_t launch_bwd_epl(const float* logits, const int32_t* idx, const float* gate,
                           const float* dgate, int s, int e, int k, int renorm, float* dlogits,
                           const DeviceInfo& di, cudaStream_t st) {
  const int threads = 256;
  long long blocks = ((long long)s * 32 + threads - 1) / threads;
  const long long cap = (long long)di.sms * 8;
  if (blocks > cap) blocks = cap;
  if (blocks < 1) blocks = 1;
  return launch_pdl(MOE_KERNEL_TOPK_GATE_BWD, topk_gate_bwd_kernel<EPL>, dim3((unsigned)blocks),
                    dim3(threads), 0, st, logits, idx, gate, dgate, s, e, k, renorm, dlogits);
}

template <int EPL>
cudaError_t launch_epl(const float* logits, int s, int e, int k, int renorm, int32_t* idx,
                       float* gate, int32_t* status, const DeviceInfo& di, cudaStream_t st) {
  const int threads = 256;
  long long blocks = ((long long)s * 32 + threads - 1) / threads;
  const long long cap = (long long)di.sms * 8;
  if (blocks > cap) blocks = cap;
  if (blocks < 1) blocks = 1;
  return launch_pdl(MOE_KERNEL_TOPK_GATE, topk_gate_kernel<EPL>, dim3((unsigned)blocks), dim3(threads), 0, st, logits, s, e,
                    k, renorm, idx, gate, status);
}

}  // namespace

cudaError_t launch_topk_gate_bwd(const float* logits, const int32_t* idx, const float* gate,
                                 const float* dgate, int s, int e, int k, int renorm,
                                 float* dlogits, const DeviceInfo& di, cudaStream_t st) {
  switch ((e + 31) / 32) {
    case 1: return launch_bwd_epl<1>(logits, idx, gate, dgate, s, e, k, renorm, dlogits, di, st);
    case 2: return launch_bwd_epl<2>(logits, idx, gate, dgate, s, e, k, renorm, dlogits, di, st);
    case 3:
    case 4: return launch_bwd_epl<4>(logits, idx, gate, dgate, s, e, k, renorm, dlogits, di, st);
    default: return launch_bwd_epl<8>(logits, idx, gate, dgate, s, e, k, renorm, dlogits, di, st);
  }
}

cudaError_t launch_topk_gate(const float* logits, int s, int e, int k, int renorm, int32_t* idx,
                             float* gate, int32_t* status, const DeviceInfo& di, cudaStream_t st) {
  const int epl = (e + 31) / 32;
  switch (epl) {
    case 1: return launch_epl<1>(logits, s, e, k, renorm, idx, gate, status, di, st);
    case 2: return launch_epl<2>(logits, s, e, k, renorm, idx, gate, status, di, st);
    case 3:
    case 4: return launch_epl<4>(logits, s, e, k, renorm, idx, gate, status, di, st);
    default: return launch_epl<8>(logits, s, e, k, renorm, idx, gate, status, di, st);
  }
}

}  // namespace moe
