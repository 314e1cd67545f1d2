// rank_slots.cu -- per-virtual-rank token-order send slots.
//
// DeepSpeed #8213 "Add an opt-in DeepEP transport for the AutoEP expert
// all-to-all", description: a token is sent to a destination rank once,
// however many of that rank's experts it selected.  Its place in the send
// buffer of rank r is its position among the tokens that go to r, in token
// order:
//   rank_slot[t,r] = #{ t' < t : token_in_rank[t',r] }   if token_in_rank[t,r]
//                  = -1                                  otherwise.
// One CTA per rank scans that rank's column of token_in_rank [s,R] (written
// by the layout kernel) in chunks of kThreads * kPerThread tokens: each
// thread counts its run of kPerThread consecutive tokens, a block-wide
// exclusive scan of the counts (warp shuffles, then the 32 warp totals)
// gives each run's first slot, and the runs are written out.  Integer-exact
// and deterministic.  Work and traffic are a few bytes per token and rank.
#include "common.cuh"
#include "internal.h"

namespace moe {

namespace {

constexpr int kThreads = 1024;
constexpr int kPerThread = 16;

__global__ void __launch_bounds__(kThreads)
    rank_slots_kernel(const uint8_t* __restrict__ tir, int s, int R, int32_t* __restrict__ slot) {
  __shared__ int s_warp[kThreads / 32];
  __shared__ int s_total;
  const int r = blockIdx.x;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  int carry = 0;  // tokens before this chunk that send to r
  for (long long c0 = 0; c0 < s; c0 += (long long)kThreads * kPerThread) {
    const long long t0 = c0 + (long long)threadIdx.x * kPerThread;
    uint32_t bits = 0;
#pragma unroll
    for (int i = 0; i < kPerThread; ++i) {
      const long long t = t0 + i;
      if (t < s && tir[t * R + r]) bits |= 1u << i;
    }
    const int n = __popc(bits);
    // inclusive scan over the warp, then over the warps
    int v = n;
#pragma unroll
    for (int d = 1; d < 32; d <<= 1) {
      const int w = __shfl_up_sync(0xffffffffu, v, d);
      if (lane >= d) v += w;
    }
    if (lane == 31) s_warp[warp] = v;
    __syncthreads();
    if (warp == 0) {
      int u = s_warp[lane];
#pragma unroll
      for (int d = 1; d < 32; d <<= 1) {
        const int w = __shfl_up_sync(0xffffffffu, u, d);
        if (lane >= d) u += w;
      }
      s_warp[lane] = u;  // inclusive prefix of the warp totals
      if (lane == 31) s_total = u;
    }
    __syncthreads();
    int next = carry + (warp > 0 ? s_warp[warp - 1] : 0) + v - n;
#pragma unroll
    for (int i = 0; i < kPerThread; ++i) {
      const long long t = t0 + i;
      if (t < s) slot[t * R + r] = ((bits >> i) & 1u) ? next++ : -1;
    }
    carry += s_total;
    __syncthreads();  // s_warp / s_total are rewritten by the next chunk
  }
}

}  // namespace

cudaError_t launch_rank_slots(const uint8_t* token_in_rank, int s, int R, int32_t* rank_slot,
                              cudaStream_t st) {
  if (s <= 0 || R <= 0) return cudaSuccess;
  rank_slots_kernel<<<R, kThreads, 0, st>>>(token_in_rank, s, R, rank_slot);
  return cudaGetLastError();
}

}  // namespace moe
