// ep.cu -- the per-rank steps of the expert-parallel exchange around the
// all-to-all: the send map with each sent row's routing metadata, and the
// gate gradients coming back.
//
// DeepSpeed #8213 "Add an opt-in DeepEP transport for the AutoEP expert
// all-to-all", description: a token goes to each destination rank once,
// not once per selected expert, and the transport replicates it itself;
// review thread: the routing weights travel with the tokens and are applied
// on the expert's rank, and their gradient must come back to the router.
//
// Rank r owns experts [r*E, (r+1)*E), E = e / R.  The send buffer holds
// the destination segments in rank order; segment r holds, in token order,
// the tokens with a kept route to rank r (the layout's send slots):
//   send_row[t, r] = (sum of rank_counts[r'] for r' < r) + rank_slot[t, r],
//                    -1 where token t sends nothing to rank r.
// With each sent row go the token's k routes as seen by the destination:
// meta_idx[q, j] = idx[t, j] - r*E when route j is kept and goes to rank r,
// else -1; meta_gate[q, j] = its gate, else 0.
#include "common.cuh"
#include "internal.h"

namespace moe {

namespace {

constexpr int kThreads = 256;
constexpr int kMaxR = 64;

// One thread per (token, destination rank): send_row[t, r] (coalesced), and
// for a sent pair its metadata row.  The token's k routes are read once per
// thread (the R threads of a token hit the same lines).
__global__ void __launch_bounds__(kThreads) ep_pack_kernel(
    const int32_t* __restrict__ idx, const int32_t* __restrict__ row, const float* __restrict__ gate,
    const int32_t* __restrict__ rank_slot, const int32_t* __restrict__ rank_counts, int s, int k, int e,
    int R, long long rows_sent, int32_t* __restrict__ send_row, int32_t* __restrict__ meta_idx,
    float* __restrict__ meta_gate, int32_t* status) {
  __shared__ long long s_off[kMaxR];
  grid_dependency_wait();
  if (threadIdx.x == 0) {
    long long run = 0;
    for (int r = 0; r < R; ++r) {
      s_off[r] = run;
      run += __ldg(rank_counts + r);
    }
  }
  __syncthreads();
  pdl_trigger_late();
  const int E = e / R;
  bool bad = false;
  const long long n = (long long)s * R;
  for (long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x; i < n; i += (long long)gridDim.x * blockDim.x) {
    const long long t = i / R;
    const int r = (int)(i - t * R);
    const int slot = __ldg(rank_slot + i);
    long long q = slot >= 0 ? s_off[r] + slot : -1;
    if (q >= rows_sent) {  // send slots that disagree with the row count given: send nothing
      bad = true;
      q = -1;
    }
    send_row[i] = (int32_t)q;
    if (q < 0) continue;
    for (int j = 0; j < k; ++j) {
      const int x = __ldg(idx + t * k + j);
      const bool on = __ldg(row + t * k + j) >= 0 && x / E == r;
      meta_idx[q * k + j] = on ? x - r * E : -1;
      meta_gate[q * k + j] = on ? __ldg(gate + t * k + j) : 0.f;
    }
  }
  if (bad) raise_status(status, MOE_DEV_BAD_ROUTE);
}

__global__ void __launch_bounds__(kThreads) ep_unpack_dgate_kernel(
    const int32_t* __restrict__ idx, const int32_t* __restrict__ row, const int32_t* __restrict__ send_row,
    const float* __restrict__ dgate_back, int s, int k, int e, int R, long long rows_sent,
    float* __restrict__ dgate) {
  grid_dependency_wait();
  pdl_trigger_late();
  const int E = e / R;
  const long long n = (long long)s * k;
  for (long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x; i < n; i += (long long)gridDim.x * blockDim.x) {
    const long long t = i / k;
    const int j = (int)(i - t * k);
    float v = 0.f;
    if (__ldg(row + i) >= 0) {
      const int r = __ldg(idx + i) / E;
      const int q = __ldg(send_row + t * R + r);
      if (q >= 0 && q < rows_sent) v = __ldg(dgate_back + (long long)q * k + j);
    }
    dgate[i] = v;
  }
}

int grid_of(long long threads, const DeviceInfo& di) {
  long long blocks = (threads + kThreads - 1) / kThreads;
  const long long cap = (long long)di.sms * 8;
  if (blocks > cap) blocks = cap;
  return (int)(blocks < 1 ? 1 : blocks);
}

}  // namespace

cudaError_t launch_ep_pack(const int32_t* idx, const int32_t* row, const float* gate, const int32_t* rank_slot,
                           const int32_t* rank_counts, int s, int k, int e, int R, long long rows_sent,
                           int32_t* send_row, int32_t* meta_idx, float* meta_gate, int32_t* status,
                           const DeviceInfo& di, cudaStream_t st) {
  return launch_pdl(MOE_KERNEL_EP_PACK, ep_pack_kernel, dim3(grid_of((long long)s * R, di)), dim3(kThreads), 0, st,
                    idx, row, gate,
                    rank_slot, rank_counts, s, k, e, R, rows_sent, send_row, meta_idx, meta_gate, status);
}

cudaError_t launch_ep_unpack_dgate(const int32_t* idx, const int32_t* row, const int32_t* send_row,
                                   const float* dgate_back, int s, int k, int e, int R, long long rows_sent,
                                   float* dgate, const DeviceInfo& di, cudaStream_t st) {
  return launch_pdl(MOE_KERNEL_EP_UNPACK, ep_unpack_dgate_kernel, dim3(grid_of((long long)s * k, di)),
                    dim3(kThreads), 0, st, idx, row, send_row, dgate_back, s, k, e, R, rows_sent, dgate);
}

}  // namespace moe
