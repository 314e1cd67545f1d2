// gate_core.cuh -- top-k softmax gating of one token by one warp.
//
// DeepSpeed #8195 "MoE dispatch: fix silent Tutel + TP corruption, speed up
// native and Tutel paths", change 1: per-route expert index and weight.
// Automodel #3684 "perf(moe): reuse the DeepEP dispatch layout on
// activation-checkpoint recompute": a recompute must route exactly as the
// forward did, so selection compares the logits themselves (no exp rounding
// can change it) and ties go to the lower expert index.
//
// Each lane holds the logits of experts lane, lane+32, ... (EPL per lane) as
// order-preserving 32-bit keys, sorted within the lane.  Each of the k rounds
// is two warp reductions (redux.sync): the largest head key, then the lowest
// expert id among the lanes holding it; that lane pops its head, and lane r
// keeps round r's winner.  The softmax max is round 0's value; the
// denominator is a butterfly sum, so every lane sees the same bits.  Used by
// the gate kernel and by the layout kernel's fused gate, so both give the
// same ids and gates.
#pragma once

#include <math.h>
#include <stdint.h>

namespace moe {

// Order-preserving 32-bit key of a float: a larger value gets a larger key,
// and -0.0 and +0.0 get the same key (adding +0.0 turns -0.0 into +0.0).
__device__ __forceinline__ uint32_t order_key(float v) {
  const uint32_t u = __float_as_uint(__fadd_rn(v, 0.0f));
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

__device__ __forceinline__ float key_value(uint32_t key) {
  return __uint_as_float((key & 0x80000000u) ? (key & 0x7fffffffu) : ~key);
}

// cur[i] = the logit of expert lane + 32*i (any value past e).  On return
// lane r < k holds the r-th selected expert in *sel_id and its gate in
// *gate_val; the return value is true on every lane when any of the token's
// e logits is NaN or infinite.
template <int EPL>
__device__ __forceinline__ bool topk_token(const float (&cur)[EPL], int lane, int e, int k, int renorm,
                                           int* sel_id_out, float* gate_out) {
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
  const bool any_bad = __any_sync(0xffffffffu, bad);
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
  *sel_id_out = sel_id;
  *gate_out = lane < k ? expf(sel_v - top) / den : 0.f;
  return any_bad;
}

}  // namespace moe

namespace moe {

// The warp's butterfly sum (xor offsets 16, 8, 4, 2, 1; each lane adds its
// partner's value to its own) of v[0..31], as one thread: IEEE addition is
// commutative, so every lane of the warp ends with exactly this tree.
__device__ __forceinline__ float butterfly_tree32(const float (&v)[32]) {
  float a[16], b[8], c[4];
#pragma unroll
  for (int i = 0; i < 16; ++i) a[i] = v[i] + v[i + 16];
#pragma unroll
  for (int i = 0; i < 8; ++i) b[i] = a[i] + a[i + 8];
#pragma unroll
  for (int i = 0; i < 4; ++i) c[i] = b[i] + b[i + 4];
  return (c[0] + c[2]) + (c[1] + c[3]);
}

// topk_token<1> (e <= 32: expert j on lane j) computed by one thread for one
// token: the same k ids in the same order (largest key first, the lower id
// on equal keys) and the same gate bits (the same expf terms, summed in the
// warp's butterfly order).  row = the token's e logits (16-byte aligned when
// e is a multiple of 4); KM >= k bounds the rounds and EM >= e (8 or 32) the
// experts, so the code a thread runs through once stays short (the terms
// past EM are zeros in the same tree).  Returns whether a logit is NaN or
// infinite.
template <int KM, int EM = 32>
__device__ __forceinline__ bool topk_token_thread(const float* __restrict__ row, int e, int k, int renorm,
                                                  int* ids, float* gates) {
  static_assert(EM == 8 || EM == 16 || EM == 32, "EM: 8, 16 or 32 experts");
  float v[32];
  if ((e & 3) == 0) {
#pragma unroll
    for (int q = 0; q < EM / 4; ++q)
      if (4 * q < e) {
        const float4 f = __ldg(reinterpret_cast<const float4*>(row) + q);
        v[4 * q] = f.x;
        v[4 * q + 1] = f.y;
        v[4 * q + 2] = f.z;
        v[4 * q + 3] = f.w;
      }
  } else {
#pragma unroll
    for (int j = 0; j < EM; ++j)
      if (j < e) v[j] = __ldg(row + j);
  }
  bool bad = false;
  uint32_t key[32];
#pragma unroll
  for (int j = 0; j < EM; ++j) {
    if (j < e && !isfinite(v[j])) bad = true;
    key[j] = j < e ? order_key(v[j]) : 0u;
  }
  uint32_t taken = 0;
  uint32_t sel_key[KM];
#pragma unroll
  for (int r = 0; r < KM; ++r) {
    sel_key[r] = 0;
    ids[r] = 0;
    if (r < k) {
      uint32_t best = 0;
      int bj = -1;
#pragma unroll
      for (int j = 0; j < EM; ++j)
        if (j < e && !((taken >> j) & 1u) && (bj < 0 || key[j] > best)) {  // equal keys keep the lower id
          best = key[j];
          bj = j;
        }
      taken |= 1u << bj;
      ids[r] = bj;
      sel_key[r] = best;
    }
  }
  const float top = key_value(sel_key[0]);
  float z[32];
#pragma unroll
  for (int j = 0; j < 32; ++j) z[j] = 0.f;
  if (renorm) {
#pragma unroll
    for (int r = 0; r < KM; ++r)
      if (r < k) z[r] = expf(key_value(sel_key[r]) - top);
  } else {
#pragma unroll
    for (int j = 0; j < EM; ++j)
      if (j < e) z[j] = expf(key_value(key[j]) - top);
  }
  const float den = butterfly_tree32(z);
#pragma unroll
  for (int r = 0; r < KM; ++r)
    if (r < k) gates[r] = (renorm ? z[r] : expf(key_value(sel_key[r]) - top)) / den;
  return bad;
}

}  // namespace moe
