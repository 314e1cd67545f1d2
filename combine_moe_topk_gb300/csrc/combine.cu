// combine.cu -- the weighted combine, its unit-weight twin (the backward of
// dispatch) and the combine backward (a gate-scaled dispatch plus the gate
// gradient).  A warp per token (or per piece of a token row when the batch
// is too short to fill the GPU), 16-byte vector loads, fp32 accumulation.
//
// DeepSpeed #8195 "MoE dispatch: fix silent Tutel + TP corruption, speed up
// native and Tutel paths", change 3: combine is a gather through the slots
// and accumulates in fp32 (as the einsum it replaces did inside the matmul).
// DeepSpeed #8213 "Add an opt-in DeepEP transport for the AutoEP expert
// all-to-all": description -- the gradient of a combine is a dispatch and the
// gradient of a dispatch is a combine; review thread -- the routing weights
// must be applied to each expert row, and their gradient must reach the
// router gate.
//
// Accumulation order is fixed: acc starts at +0.0f and takes one fmaf per
// kept route in route order, so the combine's result does not depend on the
// launch shape.  The gate gradient sums dout*y per lane in element order,
// then a butterfly across the warp, then (rows split over G warps) the G
// partial sums in warp order: fixed for a given batch shape.
#include "common.cuh"
#include "internal.h"
#include "router_grad.cuh"

namespace moe {

namespace {

constexpr int kThreads = 256;

// Tuning: 16-byte loads in flight per lane for the combine and for its
// backward (UNR = loads / KMAX),
// an optional cap on resident blocks per SM, and the width of a combine work
// unit in 16-byte vectors (0 = a whole token row per warp).
#ifndef MOE_CMB_LOADS
#define MOE_CMB_LOADS 16
#endif
#ifndef MOE_CMB_BWD_LOADS
#define MOE_CMB_BWD_LOADS 16
#endif
#ifndef MOE_CMB_MAX_BPS
#define MOE_CMB_MAX_BPS 0
#endif
#ifndef MOE_CMB_CHUNK
#define MOE_CMB_CHUNK 0
#endif
// 1: capacity layouts with k > 4 use the compacted-route kernels.
#ifndef MOE_CMB_COMPACT
#define MOE_CMB_COMPACT 1
#endif

// The gate backward fused into the combine backward: once a token's k gate
// gradients are reduced, the warp that holds them writes the token's router
// logits' gradient (router_grad_token, the gate backward kernel's own
// arithmetic).  idx = the routes' expert ids; logits only without renorm.
struct RouterGrad {
  const int32_t* idx;
  const float* logits;
  int renorm;
  float* dlogits;
};
constexpr int kRgEpl = 8;  // experts per lane covering e <= 256

// Out of line, so that the router gradient's registers are allocated on
// their own and do not change the payload loop's allocation (and hence the
// combine backward's occupancy) in the kernels that call it.
__device__ __noinline__ void router_grad_call(int t, int lane, int k, int e, const RouterGrad rg, int ij,
                                              float gj, float dgj) {
  router_grad_token<kRgEpl>(t, lane, k, e, rg.renorm, ij, gj, dgj, rg.logits, rg.dlogits);
}

// Route rows and gates of token t, broadcast from lanes 0..k-1.
// A row index outside [0, rows) counts as a dropped route: nothing past the
// buffer is read.
template <int KMAX, bool WEIGHTED>
__device__ __forceinline__ void token_routes(const int32_t* __restrict__ row,
                                             const float* __restrict__ gate, int t, int k, long long rows,
                                             int lane, int (&r)[KMAX], float (&g)[KMAX]) {
  int rl = lane < k ? __ldg(row + (size_t)t * k + lane) : -1;
  if (rl >= rows) rl = -1;
  const float gl = (WEIGHTED && lane < k) ? __ldg(gate + (size_t)t * k + lane) : 1.0f;
#pragma unroll
  for (int j = 0; j < KMAX; ++j) {
    r[j] = __shfl_sync(0xffffffffu, rl, j);
    g[j] = __shfl_sync(0xffffffffu, gl, j);
  }
}

template <typename T, int KMAX, int UNR, bool WEIGHTED>
__global__ void __launch_bounds__(kThreads) combine_kernel(const int32_t* __restrict__ row,
                                                           const float* __restrict__ gate, int s,
                                                           int k, long long rows, int nvec, int chunk, int nchunks,
                                                           const uint4* __restrict__ y,
                                                           uint4* __restrict__ out) {
  constexpr int N = Vec<T>::N;
  const int lane = threadIdx.x & 31;
  const long long warps = (gridDim.x * blockDim.x) >> 5;
  const long long units = (long long)s * nchunks;
  grid_dependency_wait();
  pdl_trigger_early();
  for (long long u = (blockIdx.x * blockDim.x + threadIdx.x) >> 5; u < units; u += warps) {
    const int t = (int)(u / nchunks);
    const int c0 = (int)(u - (long long)t * nchunks) * chunk;
    const int c1 = min(nvec, c0 + chunk);
    int r[KMAX];
    float g[KMAX];
    token_routes<KMAX, WEIGHTED>(row, gate, t, k, rows, lane, r, g);
    uint4* o = out + (size_t)t * nvec;
    for (int v0 = c0 + lane; v0 < c1; v0 += 32 * UNR) {
      uint4 val[KMAX][UNR];
#pragma unroll
      for (int j = 0; j < KMAX; ++j) {
        if (r[j] >= 0) {
          const uint4* src = y + (size_t)r[j] * nvec;
#pragma unroll
          for (int u2 = 0; u2 < UNR; ++u2) {
            const int v = v0 + 32 * u2;
            if (v < c1) val[j][u2] = ld_stream(src + v);
          }
        }
      }
#pragma unroll
      for (int u2 = 0; u2 < UNR; ++u2) {
        const int v = v0 + 32 * u2;
        if (v >= c1) break;
        float acc[N];
#pragma unroll
        for (int i = 0; i < N; ++i) acc[i] = 0.0f;
#pragma unroll
        for (int j = 0; j < KMAX; ++j) {
          if (r[j] >= 0) {
            float f[N];
            Vec<T>::to_float(val[j][u2], f);
#pragma unroll
            for (int i = 0; i < N; ++i) acc[i] = __fmaf_rn(g[j], f[i], acc[i]);
          }
        }
        st_stream(o + v, Vec<T>::from_float(acc));
      }
    }
  }
  pdl_trigger_late();
}

// Capacity layouts, where most routes may be dropped: the token's kept
// routes are first compacted onto lanes 0..nkept-1 (in route order), then
// taken KC at a time, each round loading UNR vectors of each of its routes
// and adding them into a running fp32 accumulator in route order -- the
// same fmaf sequence per element as combine_kernel, so the same bits.  The
// register tile is sized for KC routes rather than for k, so more warps fit
// and the few kept routes get more loads in flight.
template <typename T, int KC, int UNR, bool WEIGHTED>
__global__ void __launch_bounds__(kThreads) combine_compact_kernel(const int32_t* __restrict__ row,
                                                                   const float* __restrict__ gate, int s,
                                                                   int k, long long rows, int nvec, int chunk,
                                                                   int nchunks,
                                                                   const uint4* __restrict__ y,
                                                                   uint4* __restrict__ out) {
  constexpr int N = Vec<T>::N;
  const int lane = threadIdx.x & 31;
  const long long warps = (gridDim.x * blockDim.x) >> 5;
  const long long units = (long long)s * nchunks;
  grid_dependency_wait();
  pdl_trigger_early();
  for (long long u = (blockIdx.x * blockDim.x + threadIdx.x) >> 5; u < units; u += warps) {
    const int t = (int)(u / nchunks);
    const int c0 = (int)(u - (long long)t * nchunks) * chunk;
    const int c1 = min(nvec, c0 + chunk);
    int rl = lane < k ? __ldg(row + (size_t)t * k + lane) : -1;
    if (rl >= rows) rl = -1;  // past the buffer: read nothing
    const float gl = (WEIGHTED && lane < k) ? __ldg(gate + (size_t)t * k + lane) : 1.0f;
    unsigned kept = __ballot_sync(0xffffffffu, rl >= 0);
    const int nkept = __popc(kept);
    // lane c takes the c-th kept route
    int cr = -1;
    float cg = 0.f;
    for (int c = 0; kept; ++c) {  // warp-uniform: at most k rounds
      const int src = __ffs(kept) - 1;
      kept &= kept - 1u;
      const int rr = __shfl_sync(0xffffffffu, rl, src);
      const float gg = __shfl_sync(0xffffffffu, gl, src);
      if (lane == c) {
        cr = rr;
        cg = gg;
      }
    }
    uint4* o = out + (size_t)t * nvec;
    // the loop runs the same trips on every lane (the shuffles below need the
    // whole warp); a lane past the piece's end loads and stores nothing
    for (int vb = c0; vb < c1; vb += 32 * UNR) {
      const int v0 = vb + lane;
      float acc[UNR][N];
#pragma unroll
      for (int u2 = 0; u2 < UNR; ++u2)
#pragma unroll
        for (int i = 0; i < N; ++i) acc[u2][i] = 0.0f;
      for (int j0 = 0; j0 < nkept; j0 += KC) {
        int r[KC];
        float g[KC];
#pragma unroll
        for (int j = 0; j < KC; ++j) {
          r[j] = __shfl_sync(0xffffffffu, cr, (j0 + j) & 31);
          g[j] = __shfl_sync(0xffffffffu, cg, (j0 + j) & 31);
          if (j0 + j >= nkept) r[j] = -1;
        }
        uint4 val[KC][UNR];
#pragma unroll
        for (int j = 0; j < KC; ++j) {
          if (r[j] >= 0) {
            const uint4* src = y + (size_t)r[j] * nvec;
#pragma unroll
            for (int u2 = 0; u2 < UNR; ++u2) {
              const int v = v0 + 32 * u2;
              if (v < c1) val[j][u2] = ld_stream(src + v);
            }
          }
        }
#pragma unroll
        for (int u2 = 0; u2 < UNR; ++u2) {
#pragma unroll
          for (int j = 0; j < KC; ++j) {
            if (r[j] >= 0) {
              float f[N];
              Vec<T>::to_float(val[j][u2], f);
#pragma unroll
              for (int i = 0; i < N; ++i) acc[u2][i] = __fmaf_rn(g[j], f[i], acc[u2][i]);
            }
          }
        }
      }
#pragma unroll
      for (int u2 = 0; u2 < UNR; ++u2) {
        const int v = v0 + 32 * u2;
        if (v < c1) st_stream(o + v, Vec<T>::from_float(acc[u2]));
      }
    }
  }
  pdl_trigger_late();
}

// G warps per token (G = 1, 2, 4 or 8): warp w of a token's group takes the
// row's vectors [w*chunk, (w+1)*chunk); the per-route dots are reduced across
// the warp's lanes (butterfly), then across the group's warps in warp order
// through shared memory (a block-wide barrier: per-group named barriers,
// tried because the block barrier is 2.4 of 13.6 stall cycles per
// instruction on the Mixtral-like shape, made that kernel 3 % slower).
// G > 1 gives short batches more warps in flight.
template <typename T, int KMAX, int UNR, int G, bool RG>
__device__ __forceinline__ void combine_bwd_body(
    const int32_t* __restrict__ row, const int32_t* __restrict__ counts,
    const int32_t* __restrict__ offsets, long long rows, int zero_fill,
    const float* __restrict__ gate, int s, int k, int e, int nvec, int chunk,
    const uint4* __restrict__ dout, const uint4* __restrict__ y, uint4* __restrict__ dY,
    float* __restrict__ dgate, const RouterGrad& rg) {
  constexpr int N = Vec<T>::N;
  constexpr int WPB = kThreads / 32;  // warps per block
  constexpr int TPB = WPB / G;        // tokens per block and round
  __shared__ float s_dot[G > 1 ? WPB : 1][KMAX];
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int gi = warp / G, w = warp - gi * G;  // token slot in the block, warp in the group
  const int c0 = w * chunk, c1 = min(nvec, c0 + chunk);
  __shared__ SegmentStage seg;
  grid_dependency_wait();
  pdl_trigger_early();
  if (zero_fill) stage_segments_async(seg, offsets, counts, e);  // read by the zero tail
  // every warp of a block runs the same number of rounds (block-uniform loop)
  for (long long t0 = (long long)blockIdx.x * TPB; t0 < s; t0 += (long long)gridDim.x * TPB) {
    const int t = (int)(t0 + gi);
    const bool live = t < s;
    int r[KMAX];
    float g[KMAX];
    float dot[KMAX];
#pragma unroll
    for (int j = 0; j < KMAX; ++j) dot[j] = 0.0f;
    // the router gradient's own copy of the route ids and gates (lanes < k)
    int rg_id = -1;
    float rg_g = 0.f;
    if (RG && live && (G == 1 || w == 0) && lane < k) {
      rg_id = __ldg(rg.idx + (size_t)t * k + lane);
      rg_g = __ldg(gate + (size_t)t * k + lane);
    }
    if (live) {
      token_routes<KMAX, true>(row, gate, t, k, rows, lane, r, g);
      const uint4* d = dout + (size_t)t * nvec;
      for (int v0 = c0 + lane; v0 < c1; v0 += 32 * UNR) {
        uint4 dv[UNR];
        uint4 yv[KMAX][UNR];
#pragma unroll
        for (int u = 0; u < UNR; ++u) {
          const int v = v0 + 32 * u;
          if (v < c1) dv[u] = ld_stream(d + v);
        }
#pragma unroll
        for (int j = 0; j < KMAX; ++j) {
          if (r[j] >= 0) {
            const uint4* src = y + (size_t)r[j] * nvec;
#pragma unroll
            for (int u = 0; u < UNR; ++u) {
              const int v = v0 + 32 * u;
              if (v < c1) yv[j][u] = ld_stream(src + v);
            }
          }
        }
#pragma unroll
        for (int u = 0; u < UNR; ++u) {
          const int v = v0 + 32 * u;
          if (v >= c1) break;
          float df[N];
          Vec<T>::to_float(dv[u], df);
#pragma unroll
          for (int j = 0; j < KMAX; ++j) {
            if (r[j] >= 0) {
              float yf[N], p[N];
              Vec<T>::to_float(yv[j][u], yf);
#pragma unroll
              for (int i = 0; i < N; ++i) {
                dot[j] = __fmaf_rn(df[i], yf[i], dot[j]);
                p[i] = __fmul_rn(g[j], df[i]);
              }
              st_stream(dY + (size_t)r[j] * nvec + v, Vec<T>::from_float(p));
            }
          }
        }
      }
    }
    float mine = 0.0f;
#pragma unroll
    for (int j = 0; j < KMAX; ++j) {
      float v = dot[j];
#pragma unroll
      for (int off = 16; off > 0; off >>= 1) v += __shfl_xor_sync(0xffffffffu, v, off);
      if (lane == j) mine = v;
    }
    if (G == 1) {
      if (live && lane < k) dgate[(size_t)t * k + lane] = mine;
      if (RG && live) router_grad_call(t, lane, k, e, rg, rg_id, rg_g, lane < k ? mine : 0.f);
    } else {
      if (lane < KMAX) s_dot[warp][lane] = mine;
      __syncthreads();
      float sum = 0.0f;
      if (live && w == 0 && lane < k) {
#pragma unroll
        for (int q = 0; q < G; ++q) sum += s_dot[gi * G + q][lane];
        dgate[(size_t)t * k + lane] = sum;
      }
      if (RG && live && w == 0) router_grad_call(t, lane, k, e, rg, rg_id, rg_g, sum);
      __syncthreads();  // s_dot is rewritten next round
    }
  }
  pdl_trigger_late();

  // rows no kept route owns (capacity slots, padding) get zero gradient
  if (zero_fill) {
    segments_wait();  // staged since the kernel began
    const long long warps = (gridDim.x * blockDim.x) >> 5;
    const long long gw = (blockIdx.x * blockDim.x + threadIdx.x) >> 5;
    const uint4 z = make_uint4(0, 0, 0, 0);
    for (long long rr = gw; rr < rows; rr += warps) {
      if (row_is_owned(rr, seg.offsets, seg.counts, e)) continue;
      uint4* dst = dY + (size_t)rr * nvec;
      for (int v = lane; v < nvec; v += 32) st_stream(dst + v, z);
    }
  }
}

#define MOE_CBWD_PARAMS                                                                         \
  const int32_t *__restrict__ row, const int32_t *__restrict__ counts,                            \
      const int32_t *__restrict__ offsets, long long rows, int zero_fill,                         \
      const float *__restrict__ gate, int s, int k, int e, int nvec, int chunk,                   \
      const uint4 *__restrict__ dout, const uint4 *__restrict__ y, uint4 *__restrict__ dY,        \
      float *__restrict__ dgate, const RouterGrad rg
#define MOE_CBWD_ARGS row, counts, offsets, rows, zero_fill, gate, s, k, e, nvec, chunk, dout, y, dY, dgate, rg

template <typename T, int KMAX, int UNR, int G>
__global__ void __launch_bounds__(kThreads) combine_bwd_kernel(MOE_CBWD_PARAMS) {
  combine_bwd_body<T, KMAX, UNR, G, false>(MOE_CBWD_ARGS);
}

// The combine backward with the gate backward fused in: held to the plain
// kernel's two blocks per SM (128 registers) for up to 8 routes, so the
// fusion does not cost the payload loop its occupancy.
template <typename T, int KMAX, int UNR, int G>
__global__ void __launch_bounds__(kThreads, KMAX <= 8 ? 2 : 1) combine_gate_bwd_kernel(MOE_CBWD_PARAMS) {
  combine_bwd_body<T, KMAX, UNR, G, true>(MOE_CBWD_ARGS);
}
#undef MOE_CBWD_PARAMS
#undef MOE_CBWD_ARGS

// Combine backward for capacity layouts (routes may be dropped), G = 1:
// kept routes compacted onto lanes in route order and taken KC per round;
// each round walks the row (dout re-read only when a token keeps more than
// KC routes), writes dY for its routes and reduces their dots to dgate.
// Per lane the dot of a route sums the same vectors in the same order as
// combine_bwd_kernel<..., G = 1>, so dgate and dY are the same bits.
template <typename T, int KC, int UNR, bool RG>
__device__ __forceinline__ void combine_bwd_compact_body(
    const int32_t* __restrict__ row, const int32_t* __restrict__ counts,
    const int32_t* __restrict__ offsets, long long rows, int zero_fill,
    const float* __restrict__ gate, int s, int k, int e, int nvec,
    const uint4* __restrict__ dout, const uint4* __restrict__ y, uint4* __restrict__ dY,
    float* __restrict__ dgate, const RouterGrad& rg) {
  constexpr int N = Vec<T>::N;
  const int lane = threadIdx.x & 31;
  const int warps = (gridDim.x * blockDim.x) >> 5;
  const int gw = (blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  __shared__ SegmentStage seg;
  grid_dependency_wait();
  pdl_trigger_early();
  if (zero_fill) stage_segments_async(seg, offsets, counts, e);  // read by the zero tail
  for (int t = gw; t < s; t += warps) {
    int rl = lane < k ? __ldg(row + (size_t)t * k + lane) : -1;
    if (rl >= rows) rl = -1;  // past the buffer: read nothing
    const float gl = lane < k ? __ldg(gate + (size_t)t * k + lane) : 0.f;
    unsigned kept = __ballot_sync(0xffffffffu, rl >= 0);
    const int nkept = __popc(kept);
    if (lane < k && rl < 0) dgate[(size_t)t * k + lane] = 0.f;  // a dropped route
    const int rg_id = (RG && lane < k) ? __ldg(rg.idx + (size_t)t * k + lane) : -1;
    float rg_dg = 0.f;  // this lane's route's gate gradient (0 when dropped)
    // lane c takes the c-th kept route, remembering its route index
    int cr = -1, cj = 0;
    float cg = 0.f;
    for (int c = 0; kept; ++c) {  // warp-uniform: at most k rounds
      const int src = __ffs(kept) - 1;
      kept &= kept - 1u;
      const int rr = __shfl_sync(0xffffffffu, rl, src);
      const float gg = __shfl_sync(0xffffffffu, gl, src);
      if (lane == c) {
        cr = rr;
        cg = gg;
        cj = src;
      }
    }
    const uint4* d = dout + (size_t)t * nvec;
    for (int j0 = 0; j0 < nkept; j0 += KC) {
      int r[KC];
      float g[KC];
      float dot[KC];
#pragma unroll
      for (int j = 0; j < KC; ++j) {
        r[j] = __shfl_sync(0xffffffffu, cr, (j0 + j) & 31);
        g[j] = __shfl_sync(0xffffffffu, cg, (j0 + j) & 31);
        if (j0 + j >= nkept) r[j] = -1;
        dot[j] = 0.f;
      }
      for (int v0 = lane; v0 < nvec; v0 += 32 * UNR) {  // no shuffles in here
        uint4 dv[UNR];
        uint4 yv[KC][UNR];
#pragma unroll
        for (int u = 0; u < UNR; ++u) {
          const int v = v0 + 32 * u;
          if (v < nvec) dv[u] = ld_stream(d + v);
        }
#pragma unroll
        for (int j = 0; j < KC; ++j) {
          if (r[j] >= 0) {
            const uint4* src = y + (size_t)r[j] * nvec;
#pragma unroll
            for (int u = 0; u < UNR; ++u) {
              const int v = v0 + 32 * u;
              if (v < nvec) yv[j][u] = ld_stream(src + v);
            }
          }
        }
#pragma unroll
        for (int u = 0; u < UNR; ++u) {
          const int v = v0 + 32 * u;
          if (v >= nvec) break;
          float df[N];
          Vec<T>::to_float(dv[u], df);
#pragma unroll
          for (int j = 0; j < KC; ++j) {
            if (r[j] >= 0) {
              float yf[N], pp[N];
              Vec<T>::to_float(yv[j][u], yf);
#pragma unroll
              for (int i = 0; i < N; ++i) {
                dot[j] = __fmaf_rn(df[i], yf[i], dot[j]);
                pp[i] = __fmul_rn(g[j], df[i]);
              }
              st_stream(dY + (size_t)r[j] * nvec + v, Vec<T>::from_float(pp));
            }
          }
        }
      }
      // the round's dots: butterfly, then the route's own dgate slot
#pragma unroll
      for (int j = 0; j < KC; ++j) {
        float v = dot[j];
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) v += __shfl_xor_sync(0xffffffffu, v, off);
        const int jj = __shfl_sync(0xffffffffu, cj, (j0 + j) & 31);
        if (lane == 0 && j0 + j < nkept) dgate[(size_t)t * k + jj] = v;
        if (RG && lane == jj && j0 + j < nkept) rg_dg = v;
      }
    }
    if (RG) router_grad_call(t, lane, k, e, rg, rg_id, gl, rg_dg);
  }
  pdl_trigger_late();

  // rows no kept route owns (capacity slots, padding) get zero gradient
  if (zero_fill) {
    segments_wait();  // staged since the kernel began
    const uint4 z = make_uint4(0, 0, 0, 0);
    for (long long rr = gw; rr < rows; rr += warps) {
      if (row_is_owned(rr, seg.offsets, seg.counts, e)) continue;
      uint4* dst = dY + (size_t)rr * nvec;
      for (int v = lane; v < nvec; v += 32) st_stream(dst + v, z);
    }
  }
}

#define MOE_CBWDC_PARAMS                                                                        \
  const int32_t *__restrict__ row, const int32_t *__restrict__ counts,                            \
      const int32_t *__restrict__ offsets, long long rows, int zero_fill,                         \
      const float *__restrict__ gate, int s, int k, int e, int nvec,                              \
      const uint4 *__restrict__ dout, const uint4 *__restrict__ y, uint4 *__restrict__ dY,        \
      float *__restrict__ dgate, const RouterGrad rg
#define MOE_CBWDC_ARGS row, counts, offsets, rows, zero_fill, gate, s, k, e, nvec, dout, y, dY, dgate, rg

template <typename T, int KC, int UNR>
__global__ void __launch_bounds__(kThreads) combine_bwd_compact_kernel(MOE_CBWDC_PARAMS) {
  combine_bwd_compact_body<T, KC, UNR, false>(MOE_CBWDC_ARGS);
}

template <typename T, int KC, int UNR>
__global__ void __launch_bounds__(kThreads, 2) combine_gate_bwd_compact_kernel(MOE_CBWDC_PARAMS) {
  combine_bwd_compact_body<T, KC, UNR, true>(MOE_CBWDC_ARGS);
}
#undef MOE_CBWDC_PARAMS
#undef MOE_CBWDC_ARGS

// Kernel of a form: the plain combine backward, or with the gate backward fused.
template <typename T, int KMAX, int UNR, int G, bool RG>
constexpr auto cbwd_kernel() {
  if constexpr (RG) return combine_gate_bwd_kernel<T, KMAX, UNR, G>;
  else return combine_bwd_kernel<T, KMAX, UNR, G>;
}
template <typename T, int KC, int UNR, bool RG>
constexpr auto cbwd_compact_kernel() {
  if constexpr (RG) return combine_gate_bwd_compact_kernel<T, KC, UNR>;
  else return combine_bwd_compact_kernel<T, KC, UNR>;
}

template <typename K>
int occupancy(K kern) {
  int n = 0;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, kern, kThreads, 0) != cudaSuccess) return 1;
  if (MOE_CMB_MAX_BPS > 0 && n > MOE_CMB_MAX_BPS) n = MOE_CMB_MAX_BPS;
  return n;
}

// Blocks for `warps_wanted` warps of work, at most `mult` times what the SMs
// hold at once: the kernels loop over their units grid-stride, and a grid
// of a few waves -- blocks retiring and new ones starting -- measured faster
// than one resident wave looping: the combine backward 366 -> 357 us on the
// fine-grained workload at 4 waves, the combine and its unit-weight form
// 1-7 % at 2 (4 and more waves slowed the capacity and short-batch shapes).
int grid_for(long long warps_wanted, const DeviceInfo& di, int blocks_per_sm, int mult) {
  long long blocks = (warps_wanted * 32 + kThreads - 1) / kThreads;
  const long long cap = (long long)di.sms * (blocks_per_sm > 0 ? blocks_per_sm : 1) * mult;
  if (blocks > cap) blocks = cap;
  if (blocks < 1) blocks = 1;
  return (int)blocks;
}

// Pieces per token row (a power of two, 1 = whole rows) so that a short
// batch still gives `fill` times the resident warps' worth of work units;
// each piece keeps at least 32 vectors.  Measured best: fill 8 for the
// combine, 4 for its backward (whose pieces also add a shared-memory
// reduction).
int pieces_for(long long s, int nvec, const DeviceInfo& di, int blocks_per_sm, int fill, int max_pieces) {
  const long long resident = (long long)di.sms * (blocks_per_sm > 0 ? blocks_per_sm : 1) * (kThreads / 32);
  int pieces = 1;
  while (pieces < max_pieces && s * pieces < fill * resident && nvec / (2 * pieces) >= 32) pieces *= 2;
  return pieces;
}

template <typename T, int KMAX>
cudaError_t combine_t(const int32_t* row, const float* gate, int s, int k, long long rows, int m, const void* y,
                      void* out, const DeviceInfo& di, cudaStream_t st) {
  // two routes: 8 loads per lane already keep enough bytes in flight, and
  // the lower register count doubles the resident warps
  constexpr int LOADS = KMAX <= 2 ? MOE_CMB_LOADS / 2 : MOE_CMB_LOADS;
  constexpr int UNR = LOADS / KMAX > 1 ? LOADS / KMAX : 1;
  const int nvec = m / Vec<T>::N;
  auto kern_w = combine_kernel<T, KMAX, UNR, true>;
  auto kern_u = combine_kernel<T, KMAX, UNR, false>;
  static const int bps_w = occupancy(kern_w);
  static const int bps_u = occupancy(kern_u);
  const int bps = gate ? bps_w : bps_u;
  // a unit is a piece of a token row; pieces are whole multiples of 32
  // vectors so every lane has work (the sum per element is route-ordered,
  // so the split does not change any result)
  int chunk = nvec;
  if (MOE_CMB_CHUNK > 0 && MOE_CMB_CHUNK < nvec) {
    chunk = MOE_CMB_CHUNK;
  } else {
    const int pieces = pieces_for(s, nvec, di, bps, 8, 8);
    if (pieces > 1) chunk = ((nvec + pieces - 1) / pieces + 31) / 32 * 32;
  }
  const int nchunks = (nvec + chunk - 1) / chunk;
  const long long units = (long long)s * nchunks;
  if (gate)
    return launch_pdl(MOE_KERNEL_COMBINE, kern_w, dim3(grid_for(units, di, bps, 2)), dim3(kThreads), 0, st,
                      row, gate, s, k, rows, nvec, chunk, nchunks, static_cast<const uint4*>(y),
                      static_cast<uint4*>(out));
  return launch_pdl(MOE_KERNEL_DISPATCH_BWD, kern_u, dim3(grid_for(units, di, bps, 2)), dim3(kThreads), 0, st,
                    row, static_cast<const float*>(nullptr), s, k, rows, nvec, chunk, nchunks,
                    static_cast<const uint4*>(y), static_cast<uint4*>(out));
}

// y loads in flight per lane in the combine backward: half the budget with
// at most two routes or one warp per token, the full budget where several
// warps split a row of up to 8 routes (measured: the Mixtral-like backward
// 59.4 -> 56.2 us and the fine-grained one 368.8 -> 366.4 us with half, the
// stacked-replay one 51.4 -> 52.5 us).
template <int KMAX, int G>
constexpr int cbwd_unr() {
  constexpr int loads = (KMAX <= 2 || G == 1) ? MOE_CMB_BWD_LOADS / 2 : MOE_CMB_BWD_LOADS;
  return loads / KMAX > 1 ? loads / KMAX : 1;
}

template <typename T, int KMAX, int G, bool RG>
cudaError_t combine_bwd_g(const int32_t* row, const int32_t* counts, const int32_t* offsets,
                          long long rows, int zero_fill, const float* gate, int s, int k, int e,
                          int nvec, const void* dout, const void* y, void* dY, float* dgate,
                          const RouterGrad& rg, const DeviceInfo& di, int bps, cudaStream_t st) {
  constexpr int UNR = cbwd_unr<KMAX, G>();
  auto kern = cbwd_kernel<T, KMAX, UNR, G, RG>();
  const int chunk = G == 1 ? nvec : ((nvec + G - 1) / G + 31) / 32 * 32;
  long long warps = (long long)s * G;
  if (zero_fill && rows > warps) warps = rows;
  return launch_pdl(RG ? MOE_KERNEL_COMBINE_GATE_BWD : MOE_KERNEL_COMBINE_BWD, kern,
                    dim3(grid_for(warps, di, bps, 4)), dim3(kThreads), 0, st,
                    row, counts, offsets, rows, zero_fill, gate, s, k, e, nvec, chunk,
                    static_cast<const uint4*>(dout), static_cast<const uint4*>(y), static_cast<uint4*>(dY),
                    dgate, rg);
}

template <typename T, int KMAX, bool RG>
cudaError_t combine_bwd_t(const int32_t* row, const int32_t* counts, const int32_t* offsets,
                          long long rows, int zero_fill, const float* gate, int s, int k, int e,
                          int m, const void* dout, const void* y, void* dY, float* dgate, int sparse,
                          const RouterGrad& rg, const DeviceInfo& di, cudaStream_t st) {
  constexpr int UNR = cbwd_unr<KMAX, 1>();
  const int nvec = m / Vec<T>::N;
  // the split below is chosen on the plain kernel's occupancy, so the fused
  // form splits the same way and computes the same dgate bits
  static const int bps = occupancy(combine_bwd_kernel<T, KMAX, UNR, 1>);
  static const int bps_launch = occupancy(cbwd_kernel<T, KMAX, UNR, 1, RG>());
  // warps per token for short batches (the dot of the gate gradient is
  // reduced across them in a fixed order, so each G gives fixed results)
  const int G = pieces_for(s, nvec, di, bps, 4, 8);
  if (MOE_CMB_COMPACT && sparse && k > 4 && G == 1) {
    constexpr int KC = 4, UNRC = MOE_CMB_BWD_LOADS / KC > 1 ? MOE_CMB_BWD_LOADS / KC : 1;
    auto kern = cbwd_compact_kernel<T, KC, UNRC, RG>();
    static const int bpsc = occupancy(kern);
    long long warps = s;
    if (zero_fill && rows > warps) warps = rows;
    return launch_pdl(RG ? MOE_KERNEL_COMBINE_GATE_BWD : MOE_KERNEL_COMBINE_BWD, kern,
                      dim3(grid_for(warps, di, bpsc, 2)), dim3(kThreads), 0, st,
                      row, counts, offsets, rows, zero_fill, gate, s, k, e, nvec,
                      static_cast<const uint4*>(dout), static_cast<const uint4*>(y), static_cast<uint4*>(dY),
                      dgate, rg);
  }
#define MOE_CBWD_G(GG)                                                                            \
  combine_bwd_g<T, KMAX, GG, RG>(row, counts, offsets, rows, zero_fill, gate, s, k, e, nvec, dout, y, dY, \
                                 dgate, rg, di, bps_launch, st)
  if (G >= 8) return MOE_CBWD_G(8);
  if (G == 4) return MOE_CBWD_G(4);
  if (G == 2) return MOE_CBWD_G(2);
  return MOE_CBWD_G(1);
#undef MOE_CBWD_G
}

template <typename T>
cudaError_t combine_compact_t(const int32_t* row, const float* gate, int s, int k, long long rows, int m,
                              const void* y, void* out, const DeviceInfo& di, cudaStream_t st) {
  constexpr int KC = 4, UNR = 2;
  const int nvec = m / Vec<T>::N;
  auto kern_w = combine_compact_kernel<T, KC, UNR, true>;
  auto kern_u = combine_compact_kernel<T, KC, UNR, false>;
  static const int bps_w = occupancy(kern_w);
  static const int bps_u = occupancy(kern_u);
  const int bps = gate ? bps_w : bps_u;
  int chunk = nvec;
  const int pieces = pieces_for(s, nvec, di, bps, 8, 8);
  if (pieces > 1) chunk = ((nvec + pieces - 1) / pieces + 31) / 32 * 32;
  const int nchunks = (nvec + chunk - 1) / chunk;
  const long long units = (long long)s * nchunks;
  if (gate)
    return launch_pdl(MOE_KERNEL_COMBINE, kern_w, dim3(grid_for(units, di, bps, 2)), dim3(kThreads), 0, st,
                      row, gate, s, k, rows, nvec, chunk, nchunks, static_cast<const uint4*>(y),
                      static_cast<uint4*>(out));
  return launch_pdl(MOE_KERNEL_DISPATCH_BWD, kern_u, dim3(grid_for(units, di, bps, 2)), dim3(kThreads), 0, st,
                    row, static_cast<const float*>(nullptr), s, k, rows, nvec, chunk, nchunks,
                    static_cast<const uint4*>(y), static_cast<uint4*>(out));
}

template <typename T>
cudaError_t combine_k(const int32_t* row, const float* gate, int s, int k, long long rows, int m, const void* y,
                      void* out, const DeviceInfo& di, cudaStream_t st) {
  if (k <= 2) return combine_t<T, 2>(row, gate, s, k, rows, m, y, out, di, st);
  if (k <= 4) return combine_t<T, 4>(row, gate, s, k, rows, m, y, out, di, st);
  if (k <= 8) return combine_t<T, 8>(row, gate, s, k, rows, m, y, out, di, st);
  return combine_t<T, 16>(row, gate, s, k, rows, m, y, out, di, st);
}

template <typename T, bool RG>
cudaError_t combine_bwd_k(const int32_t* row, const int32_t* counts, const int32_t* offsets,
                          long long rows, int zero_fill, const float* gate, int s, int k, int e,
                          int m, const void* dout, const void* y, void* dY, float* dgate, int sparse,
                          const RouterGrad& rg, const DeviceInfo& di, cudaStream_t st) {
#define MOE_CBWD(KM)                                                                              \
  combine_bwd_t<T, KM, RG>(row, counts, offsets, rows, zero_fill, gate, s, k, e, m, dout, y, dY, dgate, \
                           sparse, rg, di, st)
  if (k <= 2) return MOE_CBWD(2);
  if (k <= 4) return MOE_CBWD(4);
  if (k <= 8) return MOE_CBWD(8);
  return MOE_CBWD(16);
#undef MOE_CBWD
}

}  // namespace

cudaError_t launch_combine(const int32_t* row, const float* gate, int s, int k, int m, int dtype,
                           const void* y, void* out, int sparse, const DeviceInfo& di, cudaStream_t st,
                           long long rows) {
  // capacity layouts (routes may be dropped) with more routes than a round holds
  if (MOE_CMB_COMPACT && sparse && k > 4) {
    if (dtype == 0) return combine_compact_t<float>(row, gate, s, k, rows, m, y, out, di, st);
    return combine_compact_t<__nv_bfloat16>(row, gate, s, k, rows, m, y, out, di, st);
  }
  if (dtype == 0) return combine_k<float>(row, gate, s, k, rows, m, y, out, di, st);
  return combine_k<__nv_bfloat16>(row, gate, s, k, rows, m, y, out, di, st);
}

cudaError_t launch_combine_bwd(const int32_t* row, const int32_t* counts, const int32_t* offsets,
                               long long rows, int zero_fill, const float* gate, int s, int k,
                               int e, int m, int dtype, const void* dout, const void* y, void* dY,
                               float* dgate, int sparse, const DeviceInfo& di, cudaStream_t st,
                               const int32_t* rg_idx, const float* rg_logits, int rg_renorm,
                               float* rg_dlogits) {
  const RouterGrad rg = {rg_idx, rg_logits, rg_renorm, rg_dlogits};
  if (rg_dlogits) {
    if (dtype == 0)
      return combine_bwd_k<float, true>(row, counts, offsets, rows, zero_fill, gate, s, k, e, m, dout, y, dY,
                                        dgate, sparse, rg, di, st);
    return combine_bwd_k<__nv_bfloat16, true>(row, counts, offsets, rows, zero_fill, gate, s, k, e, m, dout,
                                              y, dY, dgate, sparse, rg, di, st);
  }
  if (dtype == 0)
    return combine_bwd_k<float, false>(row, counts, offsets, rows, zero_fill, gate, s, k, e, m, dout, y, dY,
                                       dgate, sparse, rg, di, st);
  return combine_bwd_k<__nv_bfloat16, false>(row, counts, offsets, rows, zero_fill, gate, s, k, e, m, dout,
                                             y, dY, dgate, sparse, rg, di, st);
}

}  // namespace moe
