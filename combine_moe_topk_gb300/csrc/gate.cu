// gate.cu -- top-k softmax gating, one warp per token.
//
// DeepSpeed #8195 "MoE dispatch: fix silent Tutel + TP corruption, speed up
// native and Tutel paths", change 1: the gate hands out per-route expert
// index and weight directly (no dense [s, e] mask per route), as contiguous
// int32 routes.  Automodel #3684 "perf(moe): reuse the DeepEP dispatch
// layout on activation-checkpoint recompute": a recompute must route
// exactly as the forward did, so selection is a pure comparison on the
// logits (no exp rounding can change it) with a fixed tie-break.
//
// Each lane holds the logits of experts lane, lane+32, ... (EPL per lane).
// k rounds of a warp arg-max on (value desc, index asc) select the experts;
// lane r keeps round r's winner.  The softmax max is round 0's value; the
// denominator is a butterfly sum, so every lane sees the same bits.
#include <math.h>

#include "common.cuh"
#include "internal.h"

namespace moe {

namespace {

__device__ __forceinline__ bool before(float av, int ai, float bv, int bi) {
  return av > bv || (av == bv && ai < bi);
}

template <int EPL>
__global__ void __launch_bounds__(256) topk_gate_kernel(const float* __restrict__ logits, int s,
                                                        int e, int k, int renorm,
                                                        int32_t* __restrict__ idx,
                                                        float* __restrict__ gate,
                                                        int32_t* status) {
  const int lane = threadIdx.x & 31;
  const int warps = (gridDim.x * blockDim.x) >> 5;
  for (int t = (blockIdx.x * blockDim.x + threadIdx.x) >> 5; t < s; t += warps) {
    const float* l = logits + (size_t)t * e;
    float v[EPL];
    bool bad = false;
#pragma unroll
    for (int i = 0; i < EPL; ++i) {
      const int j = lane + 32 * i;
      v[i] = j < e ? __ldg(l + j) : -INFINITY;  // padding is never selected: k <= e
      if (j < e && !isfinite(v[i])) bad = true;
    }
    if (__any_sync(0xffffffffu, bad)) {
      if (lane == 0) raise_status(status, MOE_DEV_NONFINITE);
    }

    unsigned taken = 0;
    float sel_v = -INFINITY;  // lane r < k: the r-th selected logit
    int sel_i = 0;
    float top = 0.f;
    for (int r = 0; r < k; ++r) {
      float bv = -INFINITY;
      int bi = 0x7fffffff;
#pragma unroll
      for (int i = 0; i < EPL; ++i) {
        const int j = lane + 32 * i;
        if (!((taken >> i) & 1u) && before(v[i], j, bv, bi)) {
          bv = v[i];
          bi = j;
        }
      }
#pragma unroll
      for (int off = 16; off > 0; off >>= 1) {
        const float ov = __shfl_xor_sync(0xffffffffu, bv, off);
        const int oi = __shfl_xor_sync(0xffffffffu, bi, off);
        if (before(ov, oi, bv, bi)) {
          bv = ov;
          bi = oi;
        }
      }
      if ((bi & 31) == lane && bi < 32 * EPL) taken |= 1u << (bi >> 5);
      if (lane == r) {
        sel_v = bv;
        sel_i = bi;
      }
      if (r == 0) top = bv;
    }

    float z = 0.f;
    if (renorm) {
      if (lane < k) z = expf(sel_v - top);
    } else {
#pragma unroll
      for (int i = 0; i < EPL; ++i)
        if (lane + 32 * i < e) z += expf(v[i] - top);
    }
    float den = z;
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) den += __shfl_xor_sync(0xffffffffu, den, off);
    if (lane < k) {
      idx[(size_t)t * k + lane] = sel_i;
      gate[(size_t)t * k + lane] = expf(sel_v - top) / den;
    }
  }
}

template <int EPL>
cudaError_t launch_epl(const float* logits, int s, int e, int k, int renorm, int32_t* idx,
                       float* gate, int32_t* status, const DeviceInfo& di, cudaStream_t st) {
  const int threads = 256;
  long long blocks = ((long long)s * 32 + threads - 1) / threads;
  const long long cap = (long long)di.sms * 8;
  if (blocks > cap) blocks = cap;
  if (blocks < 1) blocks = 1;
  (void)cudaGetLastError();  // clear a stale error left by an earlier, unrelated call
  topk_gate_kernel<EPL><<<(int)blocks, threads, 0, st>>>(logits, s, e, k, renorm, idx, gate, status);
  return cudaGetLastError();
}

}  // namespace

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
