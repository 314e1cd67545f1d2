// dispatch.cu -- gather token rows into the expert-grouped buffer.
//
// DeepSpeed #8195 "MoE dispatch: fix silent Tutel + TP corruption, speed up
// native and Tutel paths", change 3: route each token through its slot
// directly, so dispatch is one gather moving s*k rows instead of a dense
// [s, e, c] einsum; change 2: the capacity buffer is [e, c, m] (row
// x*c + slot), never a flat buffer sliced along the wrong dimension.
// DeepSpeed #8213 "Add an opt-in DeepEP transport for the AutoEP expert
// all-to-all", description: the dispatch takes tokens before top-k
// expansion and replicates them itself -- here each token row is read from
// HBM once and written to each of its kept routes.
//
// A warp per token, or per piece of a token row when the batch is short of
// 8x the resident warps.  Each lane loads UNR 16-byte vectors of the piece
// (all loads in flight before the first store), then stores them to every
// kept route's row: each store instruction writes 512 contiguous bytes.
// The routes are read by lanes 0..k-1 and broadcast by shuffle; a token
// with no kept route reads nothing.  Rows no route owns (capacity slots
// past the counts, per-expert padding) are zeroed afterwards, a warp per
// row, against the segments the block stages in shared memory meanwhile.
// Nothing waits on anything but the previous kernel (the programmatic
// launch dependency), so the kernel has no time-out path.
//
// An earlier form moved the rows with 1-D bulk (TMA) copies through a
// shared-memory ring, one warp per CTA; at the same bytes it was 9 % slower
// on the GShard capacity workload and 25 % slower on the 256-token one,
// and no faster elsewhere.
#include "common.cuh"
#include "internal.h"

namespace moe {

namespace {

// Tuning: 16-byte vectors in flight per lane, cap on CTAs (of 256 threads)
// per SM below what the registers allow.
#ifndef MOE_DSP_UNR
#define MOE_DSP_UNR 8
#endif
#ifndef MOE_DSP_BPS
#define MOE_DSP_BPS 8
#endif

// KMAX: routes per token rounded up to a power of two (k, or the ranks of an
// expert-parallel send, at most 32).  A unit is (token, piece); a piece is
// `chunk` vectors of the row, a multiple of 32.
template <int KMAX, int UNR>
__global__ void __launch_bounds__(256) dispatch_kernel(
    const int32_t* __restrict__ row, const int32_t* __restrict__ counts, const int32_t* __restrict__ offsets,
    int s, int k, int e, long long rows, int zero_fill, int nvec, int chunk, int nchunks,
    const uint4* __restrict__ x, uint4* __restrict__ X, int32_t* status) {
  const int lane = threadIdx.x & 31;
  const long long warps = ((long long)gridDim.x * blockDim.x) >> 5;
  const long long gw = ((long long)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  const long long units = (long long)s * nchunks;
  __shared__ SegmentStage seg;
  grid_dependency_wait();
  pdl_trigger_early();
  if (zero_fill) stage_segments_async(seg, offsets, counts, e);  // read by the zero tail
  bool bad = false;
  for (long long u = gw; u < units; u += warps) {
    const int t = (int)(u / nchunks);
    const int c0 = (int)(u - (long long)t * nchunks) * chunk;
    const int c1 = min(nvec, c0 + chunk);
    int rl = lane < k ? __ldg(row + (size_t)t * k + lane) : -1;
    if (rl >= rows) {  // a row past the buffer: written nowhere, reported
      bad = true;
      rl = -1;
    }
    if (!__any_sync(0xffffffffu, rl >= 0)) continue;  // every route dropped: nothing to read
    int r[KMAX];
#pragma unroll
    for (int j = 0; j < KMAX; ++j) r[j] = __shfl_sync(0xffffffffu, rl, j);
    const uint4* src = x + (size_t)t * nvec;
    for (int v0 = c0 + lane; v0 < c1; v0 += 32 * UNR) {
      uint4 val[UNR];
#pragma unroll
      for (int q = 0; q < UNR; ++q) {
        const int v = v0 + 32 * q;
        if (v < c1) val[q] = ld_stream(src + v);
      }
#pragma unroll
      for (int j = 0; j < KMAX; ++j) {
        if (j < k && r[j] >= 0) {
          uint4* dst = X + (size_t)r[j] * nvec;
#pragma unroll
          for (int q = 0; q < UNR; ++q) {
            const int v = v0 + 32 * q;
            if (v < c1) st_stream(dst + v, val[q]);
          }
        }
      }
    }
  }
  pdl_trigger_late();
  if (bad) raise_status(status, MOE_DEV_BAD_ROUTE);
  if (zero_fill) {
    segments_wait();  // staged since the kernel began
    const uint4 z = make_uint4(0, 0, 0, 0);
    for (long long rr = gw; rr < rows; rr += warps) {
      if (row_is_owned(rr, seg.offsets, seg.counts, e)) continue;
      uint4* dst = X + (size_t)rr * nvec;
      for (int v = lane; v < nvec; v += 32) st_stream(dst + v, z);
    }
  }
}

template <int KMAX>
cudaError_t launch(const int32_t* row, const int32_t* counts, const int32_t* offsets, int s, int k, int e,
                   long long rows, int zero_fill, const void* x, void* X, long long row_bytes, int32_t* status,
                   const DeviceInfo& di, cudaStream_t st) {
  auto kern = dispatch_kernel<KMAX, MOE_DSP_UNR>;
  static OncePerDevice occ_once;
  static int bps[kOnceDevices];
  int dev = 0;
  cudaError_t err = cudaGetDevice(&dev);
  if (err != cudaSuccess) return err;
  err = occ_once.run([&] {
    int n = 0;
    cudaError_t e2 = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, kern, 256, 0);
    if (n > MOE_DSP_BPS) n = MOE_DSP_BPS;
    if (e2 == cudaSuccess) bps[dev] = n < 1 ? 1 : n;
    return e2;
  });
  if (err != cudaSuccess) return err;
  const int nvec = (int)(row_bytes / 16);
  // pieces of a row (a power of two, each at least 32 vectors) while the
  // units number fewer than 8x the resident warps
  const long long resident = (long long)di.sms * bps[dev] * 8;
  int pieces = 1;
  while (pieces < 8 && (long long)s * pieces < 8 * resident && nvec / (2 * pieces) >= 32) pieces *= 2;
  const int chunk = pieces > 1 ? ((nvec + pieces - 1) / pieces + 31) / 32 * 32 : nvec;
  const int nchunks = (nvec + chunk - 1) / chunk;
  long long warps = (long long)s * nchunks;
  if (zero_fill && rows > warps) warps = rows;
  long long blocks = (warps * 32 + 255) / 256;
  // up to 16 waves of blocks (in practice a warp per unit): blocks that
  // retire and make room for new ones measured faster than one resident wave
  // looping over the units -- 202 -> 181 us on the fine-grained workload,
  // 146 -> 135 us on the GShard-like one
  const long long cap = (long long)di.sms * bps[dev] * 16;
  if (blocks > cap) blocks = cap;
  if (blocks < 1) blocks = 1;
  return launch_pdl(MOE_KERNEL_DISPATCH, kern, dim3((unsigned)blocks), dim3(256), 0, st, row, counts, offsets, s, k,
                    e, rows, zero_fill, nvec, chunk, nchunks, static_cast<const uint4*>(x), static_cast<uint4*>(X),
                    status);
}

}  // namespace

cudaError_t launch_dispatch(const int32_t* row, const int32_t* counts, const int32_t* offsets, int s,
                            int k, int e, long long rows, int zero_fill, const void* x,
                            void* X, long long row_bytes, int32_t* status, const DeviceInfo& di,
                            cudaStream_t st) {
  if (k <= 2) return launch<2>(row, counts, offsets, s, k, e, rows, zero_fill, x, X, row_bytes, status, di, st);
  if (k <= 4) return launch<4>(row, counts, offsets, s, k, e, rows, zero_fill, x, X, row_bytes, status, di, st);
  if (k <= 8) return launch<8>(row, counts, offsets, s, k, e, rows, zero_fill, x, X, row_bytes, status, di, st);
  if (k <= 16) return launch<16>(row, counts, offsets, s, k, e, rows, zero_fill, x, X, row_bytes, status, di, st);
  return launch<32>(row, counts, offsets, s, k, e, rows, zero_fill, x, X, row_bytes, status, di, st);
}

}  // namespace moe
