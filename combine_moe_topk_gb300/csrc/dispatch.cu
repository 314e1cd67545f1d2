// dispatch.cu -- gather token rows into the expert-grouped buffer with 1-D
// bulk (TMA) copies staged through shared memory.
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
// One warp per CTA, several CTAs per SM, each CTA owning a contiguous token
// range.  A ring of `stages` shared-memory buffers: lane 0 loads a token row
// (or a piece of it) with cp.async.bulk global->shared, completion counted
// on the stage's mbarrier; once it lands, lane j issues the bulk
// shared->global store for route j, and every lane commits one bulk group
// per unit, so `wait_group.read 1` tells when the previous unit's buffer may
// be refilled.  In capacity mode the CTA then writes the zero tail of its
// share of the [e, c] slots from a zeroed buffer.  All mbarrier waits are
// bounded; on time-out the kernel records MOE_DEV_TIMEOUT, waits (bounded)
// for its loads in flight and for its stores, and returns.
#include "common.cuh"
#include "internal.h"

namespace moe {

namespace {

// Tuning: ring depth, largest bulk piece in bytes, cap on CTAs per SM.
#ifndef MOE_DSP_STAGES
#define MOE_DSP_STAGES 4
#endif
#ifndef MOE_DSP_PIECE
#define MOE_DSP_PIECE 16384
#endif
#ifndef MOE_DSP_MAX_CTAS
#define MOE_DSP_MAX_CTAS 16
#endif

constexpr int kMaxStages = MOE_DSP_STAGES;
constexpr int kBatch = 32;       // tokens of routing metadata staged at a time (at most)
constexpr int kMaxK = 32;        // routes per token: k, or the ranks of an expert-parallel send
constexpr int kRowBudget = 512;  // staged route rows: a batch holds min(32, 512 / k) tokens
constexpr int kMaxE = 256;
// The static shared memory stays under 5 KB so that six CTAs with a 4-stage
// ring of 8 KB rows fit on an SM (at 7.4 KB, with 32 x 32 staged routes, only
// five did: 2 % of the dispatch's time on the fine-grained workload).

struct Params {
  const char* x;
  char* X;
  const int32_t* row;
  const int32_t* counts;
  const int32_t* offsets;
  int s, k, e, capacity;
  long long rows;   // rows of X
  int zero_fill;    // X has rows no route owns (capacity slots, padding): zero them
  long long row_bytes;
  int piece;       // bytes per unit (multiple of 16)
  int npieces;     // units per token row
  int stages;
  int stage_stride;
  int32_t* status;
  long long timeout_ns;
};

__global__ void __launch_bounds__(32) dispatch_kernel(const Params p) {
  extern __shared__ __align__(128) unsigned char buf[];
  __shared__ __align__(8) uint64_t bar[kMaxStages];
  __shared__ int desc_rows[kMaxStages][kMaxK];
  __shared__ int desc_t[kMaxStages];
  __shared__ int desc_p[kMaxStages];
  __shared__ int b_rows[kRowBudget];
  __shared__ unsigned b_mask[kBatch];
  __shared__ int s_counts[kMaxE];
  __shared__ int s_offsets[kMaxE + 1];

  const int lane = threadIdx.x;
  const long long G = gridDim.x, b = blockIdx.x;
  const int t0 = (int)((long long)p.s * b / G);
  const int t1 = (int)((long long)p.s * (b + 1) / G);
  const uint64_t deadline = globaltimer_ns() + (uint64_t)p.timeout_ns;

  if (lane == 0) {
    for (int st = 0; st < p.stages; ++st) mbar_init(&bar[st], 1);
    fence_barrier_init();
  }
  grid_dependency_wait();
  pdl_trigger_early();
  if (p.zero_fill) {
    for (int x = lane; x < p.e; x += 32) s_counts[x] = __ldg(p.counts + x);
    for (int x = lane; x <= p.e; x += 32) s_offsets[x] = __ldg(p.offsets + x);
  }
  __syncwarp();

  // ---- unit iterator (uniform across the warp) ----------------------------
  int tb = t0, blen = 0, ti = 0, pi = 0;
  auto next_unit = [&](int st) -> bool {
    for (;;) {
      if (ti == blen) {
        tb += blen;
        if (tb >= t1) return false;
        blen = min(min(kBatch, kRowBudget / p.k), t1 - tb);
        ti = 0;
        pi = 0;
        __syncwarp();
        for (int i = lane; i < blen * p.k; i += 32) b_rows[i] = __ldg(p.row + (size_t)tb * p.k + i);
        __syncwarp();
        if (lane < blen) {
          unsigned mk = 0;
          for (int j = 0; j < p.k; ++j) {
            const int r = b_rows[lane * p.k + j];
            if (r >= 0 && r < p.rows) {
              mk |= 1u << j;
            } else if (r >= 0) {  // a row past the buffer: written nowhere, reported
              b_rows[lane * p.k + j] = -1;
              raise_status(p.status, MOE_DEV_BAD_ROUTE);
            }
          }
          b_mask[lane] = mk;
        }
        __syncwarp();
      }
      if (b_mask[ti] == 0) {  // every route of this token was dropped
        ++ti;
        continue;
      }
      break;
    }
    const int t = tb + ti;
    const int pc = pi;
    if (lane < p.k) desc_rows[st][lane] = b_rows[ti * p.k + lane];
    if (lane == 0) {
      desc_t[st] = t;
      desc_p[st] = pc;
    }
    __syncwarp();
    if (lane == 0) {
      const long long off = (long long)pc * p.piece;
      const uint32_t bytes = (uint32_t)min((long long)p.piece, p.row_bytes - off);
      mbar_arrive_expect_tx(&bar[st], bytes);
      bulk_g2s(buf + (size_t)st * p.stage_stride, p.x + (size_t)t * p.row_bytes + off, bytes,
               &bar[st]);
    }
    if (++pi == p.npieces) {
      pi = 0;
      ++ti;
    }
    return true;
  };

  // ---- pipeline -------------------------------------------------------------
  long long issued = 0, done = 0;
  for (int st = 0; st < p.stages; ++st) {
    if (!next_unit(st)) break;
    ++issued;
  }
  uint32_t parity = 0;
  bool ok = true;
  while (done < issued) {
    const int st = (int)(done % p.stages);
    if (!mbar_wait_bounded(&bar[st], (parity >> st) & 1u, deadline)) {
      ok = false;
      break;
    }
    parity ^= 1u << st;
    const int t = desc_t[st];
    const long long off = (long long)desc_p[st] * p.piece;
    const uint32_t bytes = (uint32_t)min((long long)p.piece, p.row_bytes - off);
    (void)t;
    if (lane < p.k) {
      const int r = desc_rows[st][lane];
      if (r >= 0) bulk_s2g(p.X + (size_t)r * p.row_bytes + off, buf + (size_t)st * p.stage_stride, bytes);
    }
    bulk_commit();
    if (done >= 1) {
      // the unit before this one has finished reading its buffer: refill it
      bulk_wait_read<1>();
      __syncwarp();
      const int prev = (int)((done - 1) % p.stages);
      if (next_unit(prev)) ++issued;
    }
    ++done;
  }

  if (!ok) {
    pdl_trigger_late();
    if (lane == 0) raise_status(p.status, MOE_DEV_TIMEOUT);
    // let the loads still in flight land before the CTA's shared memory goes
    const uint64_t drain = globaltimer_ns() + (uint64_t)p.timeout_ns;
    for (long long u = done; u < issued; ++u) {
      const int st = (int)(u % p.stages);
      if (!mbar_wait_bounded(&bar[st], (parity >> st) & 1u, drain)) break;
      parity ^= 1u << st;
    }
    bulk_wait_all();
    return;
  }

  pdl_trigger_late();
  // ---- rows no route owns: capacity slots past counts, padding ------------
  if (p.zero_fill) {
    bulk_wait_all();
    __syncwarp();
    uint4* z = reinterpret_cast<uint4*>(buf);
    for (int i = lane; i < p.stage_stride / 16; i += 32) z[i] = make_uint4(0, 0, 0, 0);
    fence_proxy_async_smem();
    __syncwarp();
    const long long r0 = p.rows * b / G, r1 = p.rows * (b + 1) / G;
    for (long long r = r0 + lane; r < r1; r += 32) {
      if (row_is_owned(r, s_offsets, s_counts, p.e)) continue;
      for (int pc = 0; pc < p.npieces; ++pc) {
        const long long off = (long long)pc * p.piece;
        const uint32_t bytes = (uint32_t)min((long long)p.piece, p.row_bytes - off);
        bulk_s2g(p.X + (size_t)r * p.row_bytes + off, buf, bytes);
      }
    }
    bulk_commit();
  }
  bulk_wait_all();
}


struct Config {
  int piece, npieces, stages, stride, smem, ctas_per_sm;
};

Config choose(long long row_bytes) {
  Config c;
  const long long kPieceMax = MOE_DSP_PIECE;
  c.npieces = (int)((row_bytes + kPieceMax - 1) / kPieceMax);
  long long piece = (row_bytes + c.npieces - 1) / c.npieces;
  piece = (piece + 15) / 16 * 16;
  c.piece = (int)piece;
  c.stride = (int)((piece + 127) / 128 * 128);
  c.stages = MOE_DSP_STAGES;
  c.smem = c.stages * c.stride;
  int n = 0;
  cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, dispatch_kernel, 32, c.smem);
  c.ctas_per_sm = n < 1 ? 1 : (n > MOE_DSP_MAX_CTAS ? MOE_DSP_MAX_CTAS : n);
  return c;
}

}  // namespace

cudaError_t launch_dispatch(const int32_t* row, const int32_t* counts, const int32_t* offsets, int s,
                            int k, int e, int capacity, long long rows, int zero_fill, const void* x,
                            void* X, long long row_bytes, int32_t* status, const DeviceInfo& di,
                            cudaStream_t st) {
  // allow the kernel the device's whole opt-in shared memory (less its static
  // part) once per device; occupancy still follows the dynamic size launched
  static OncePerDevice opt_in;
  cudaError_t err = opt_in.run([&] {
    cudaFuncAttributes fa;
    cudaError_t e = cudaFuncGetAttributes(&fa, dispatch_kernel);
    if (e == cudaSuccess)
      e = cudaFuncSetAttribute(dispatch_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                               di.max_smem_optin - (int)fa.sharedSizeBytes);
    return e;
  });
  if (err != cudaSuccess) return err;
  Config c = choose(row_bytes);
  Params p;
  p.x = static_cast<const char*>(x);
  p.X = static_cast<char*>(X);
  p.row = row;
  p.counts = counts;
  p.offsets = offsets;
  p.rows = rows;
  p.zero_fill = zero_fill;
  p.s = s;
  p.k = k;
  p.e = e;
  p.capacity = capacity;
  p.row_bytes = row_bytes;
  p.piece = c.piece;
  p.npieces = c.npieces;
  p.stages = c.stages;
  p.stage_stride = c.stride;
  p.status = status;
  p.timeout_ns = 2000000000LL;

  long long work = s;
  if (zero_fill) {
    const long long zero_groups = (rows + 31) / 32;
    if (zero_groups > work) work = zero_groups;
  }
  long long grid = (long long)di.sms * c.ctas_per_sm;
  if (grid > work) grid = work;
  if (grid < 1) grid = 1;
  return launch_pdl(MOE_KERNEL_DISPATCH, dispatch_kernel, dim3((unsigned)grid), dim3(32), (size_t)c.smem, st, p);
}

}  // namespace moe
