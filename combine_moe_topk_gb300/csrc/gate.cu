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
// Each lane holds the logits of experts lane, lane+32, ... (EPL per lane) as
// order-preserving 32-bit keys, sorted within the lane.  Each of the k rounds
// is two warp reductions (redux.sync): the largest head key, then the lowest
// expert id among the lanes holding it; that lane pops its head, and lane r
// keeps round r's winner.  The softmax max is round 0's value; the
// denominator is a butterfly sum, so every lane sees the same bits.
#include <math.h>

#include "common.cuh"
#include "internal.h"
#include "router_grad.cuh"

namespace moe {

namespace {

// Order-preserving 32-bit key of a float: a larger value gets a larger key,
// and -0.0 and +0.0 get the same key (adding +0.0 turns -0.0 into +0.0).
__device__ __forceinline__ uint32_t order_key(float v) {
  const uint32_t u = __float_as_uint(__fadd_rn(v, 0.0f));
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

__device__ __forceinline__ float key_value(uint32_t key) {
  return __uint_as_float((key & 0x80000000u) ? (key & 0x7fffffffu) : ~key);
}

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
    // this lane's candidates, experts lane + 32*i; key 0 marks padding (below -inf)
    uint32_t key[EPL];
    int id[EPL];
    bool bad = false;
#pragma unroll
    for (int i = 0; i < EPL; ++i) {
      const int j = lane + 32 * i;
      const float v = cur[i];
      if (j < e && !isfinite(v)) bad = true;
      key[i] = j < e ? order_key(v) : 0u;
      id[i] = j;
    }
    if (__any_sync(0xffffffffu, bad) && lane == 0) raise_status(status, MOE_DEV_NONFINITE);
    // stable sort of the lane's candidates, largest key first (equal keys keep
    // their ascending expert order)
#pragma unroll
    for (int a = 0; a < EPL; ++a)
#pragma unroll
      for (int b = EPL - 1; b > a; --b)
        if (key[b] > key[b - 1]) {
          const uint32_t tk = key[b];
          key[b] = key[b - 1];
          key[b - 1] = tk;
          const int ti = id[b];
          id[b] = id[b - 1];
          id[b - 1] = ti;
        }
    // the lane's values, kept for the full-softmax sum before the selection
    // consumes them; the first `nvalid` sorted entries are real experts
    const int nvalid = min(EPL, max(0, (e - lane + 31) / 32));
    float all_v[EPL];
#pragma unroll
    for (int i = 0; i < EPL; ++i) all_v[i] = key_value(key[i]);
    uint32_t top_key = 0;
    uint32_t sel_key = 0;
    int sel_id = 0;
    // k rounds: the warp's largest head key, ties to the lower expert id
    for (int r = 0; r < k; ++r) {
      const uint32_t m = __reduce_max_sync(0xffffffffu, key[0]);
      const uint32_t cand = key[0] == m ? (uint32_t)id[0] : 0xffffffffu;
      const uint32_t j = __reduce_min_sync(0xffffffffu, cand);
      if (key[0] == m && (uint32_t)id[0] == j) {  // the winner pops its head
#pragma unroll
        for (int i = 0; i + 1 < EPL; ++i) {
          key[i] = key[i + 1];
          id[i] = id[i + 1];
        }
        key[EPL - 1] = 0u;
      }
      if (lane == r) {
        sel_key = m;
        sel_id = (int)j;
      }
      if (r == 0) top_key = m;
    }
    const float top = key_value(top_key);
    const float sel_v = key_value(sel_key);

    float z = 0.f;
    if (renorm) {
      if (lane < k) z = expf(sel_v - top);
    } else {
#pragma unroll
      for (int i = 0; i < EPL; ++i)
        if (i < nvalid) z += expf(all_v[i] - top);
    }
    float den = z;
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) den += __shfl_xor_sync(0xffffffffu, den, off);
    if (lane < k) {
      idx[(size_t)t * k + lane] = sel_id;
      gate[(size_t)t * k + lane] = expf(sel_v - top) / den;
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
