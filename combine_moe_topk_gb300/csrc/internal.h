// internal.h -- host-side launchers of the kernels, called by api.cu after
// argument validation.  Each returns the cudaError_t of its launch.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include <mutex>

namespace moe {

// Runs `set_up` (returning a cudaError_t) once per device, thread-safe, and
// hands every later caller the same result.  For per-device one-time steps
// such as a kernel's shared-memory opt-in.
constexpr int kOnceDevices = 64;
struct OncePerDevice {
  std::once_flag flag[kOnceDevices];
  cudaError_t result[kOnceDevices] = {};
  template <class F>
  cudaError_t run(F&& set_up) {
    int dev = 0;
    cudaError_t err = cudaGetDevice(&dev);
    if (err != cudaSuccess) return err;
    if (dev < 0 || dev >= kOnceDevices) return cudaErrorInvalidDevice;
    std::call_once(flag[dev], [&] { result[dev] = set_up(); });
    return result[dev];
  }
};

struct DeviceInfo {
  int sms = 0;                 // streaming multiprocessors
  int layout_blocks_per_sm = 0;
  int gate_layout_blocks_per_sm = 0;  // the layout kernel with the gate fused in
  int max_smem_optin = 0;      // bytes of dynamic shared memory a block may opt into
};

const DeviceInfo& device_info(int device);

// --- gate ---------------------------------------------------------------
cudaError_t launch_topk_gate(const float* logits, int s, int e, int k, int renorm, int32_t* idx,
                             float* gate, int32_t* status, const DeviceInfo& di, cudaStream_t st);

cudaError_t launch_topk_gate_bwd(const float* logits, const int32_t* idx, const float* gate,
                                 const float* dgate, int s, int e, int k, int renorm,
                                 float* dlogits, const DeviceInfo& di, cudaStream_t st);

// --- layout -------------------------------------------------------------
struct LayoutPlan {
  int tiles = 1;            // CTAs (all co-resident: cooperative launch)
  int subtiles_per_tile = 1;
};
LayoutPlan plan_layout(int s, int e, const DeviceInfo& di);
size_t lookback_bytes(const LayoutPlan& plan, int e);  // scratch the plan's look-back needs
int layout_blocks_per_sm();                            // co-resident layout CTAs per SM

struct LayoutOut {
  int32_t* idx;
  int32_t* loc;
  int32_t* row;
  uint8_t* drop;
  int32_t* raw_counts;
  int32_t* counts;
  int32_t* offsets;
  uint8_t* token_in_rank;
  int32_t* rank_counts;
  unsigned* lookback;            // [tiles][e rounded up to 4], zero before the launch
  int32_t* status;
  int32_t* inv_row = nullptr;    // [rows]: token of each kept route's row (optional)
};

// One build of a layout into its arrays (the look-back words must have been
// zeroed once, or left by an earlier build of the same plan: the kernel
// takes the other parity from each tile's own row).  clear_status: the
// kernel itself zeroes the status word and the rank counts (so a rebuild
// needs no memset).  logits != nullptr: the top-k gate runs fused in the
// same kernel (renorm; the ids to gate_idx, the gates to gate_val); only
// when layout_can_fuse_gate(plan, priority, e, di).
struct LayoutBuild {
  int clear_status = 0;
  int absent_ok = 0;  // expert id -1 = no route (row -1, drop 1, no status bit)
  const float* logits = nullptr;
  int renorm = 1;
  int32_t* gate_idx = nullptr;
  float* gate_val = nullptr;
};
bool layout_can_fuse_gate(const LayoutPlan& plan, int priority, int e, const DeviceInfo& di);
int gate_layout_blocks_per_sm();

// priority 0 = token order, 1 = k-major; pad_multiple >= 1 pads dropless
// expert segments.  The plan must be made for s units (s * k when k-major).
// rows: the dispatched buffer's rows; a dropless route whose row would fall at
// or past it gets none (MOE_DEV_ROWS_EXCEEDED), and counts / offsets are cut there.
cudaError_t launch_layout(const int32_t* topk_idx, int s, int e, int k, int capacity, int R,
                          int priority, int pad_multiple, int rows, const LayoutPlan& plan,
                          const LayoutOut& out, int hold_tile, long long timeout_ns,
                          cudaStream_t st, const LayoutBuild& build);

// Allocation-free layout: the look-back scratch is a file-scope device array
// of noalloc_lookback_words() words; returns cudaErrorInvalidValue (and sets
// *words_needed) when tiles * e exceeds it.  out.lookback is ignored.
int noalloc_lookback_words();
cudaError_t launch_layout_noalloc(const int32_t* topk_idx, int s, int e, int k, int capacity, int R,
                                  const LayoutOut& out, int* words_needed, cudaStream_t st);

// --- dispatch (register-staged gather) -----------------------------------
// zero_fill: X has rows no route owns (capacity slots past the count,
// per-expert padding); they are written with zeros.
cudaError_t launch_dispatch(const int32_t* row, const int32_t* counts, const int32_t* offsets, int s,
                            int k, int e, long long rows, int zero_fill, const void* x,
                            void* X, long long row_bytes, int32_t* status, const DeviceInfo& di,
                            cudaStream_t st);

// --- combine family -----------------------------------------------------
// dtype: 0 = f32, 1 = bf16.  gate == nullptr means unit weights.
// sparse: the layout may have dropped routes (capacity mode)
// rows: rows of y; a row index at or past it counts as a dropped route.
cudaError_t launch_combine(const int32_t* row, const float* gate, int s, int k, int m, int dtype,
                           const void* y, void* out, int sparse, const DeviceInfo& di, cudaStream_t st,
                           long long rows);

// With rg_dlogits != nullptr the top-k gate backward runs fused into the
// same kernel (rg_idx = the routes' expert ids; rg_logits only when
// rg_renorm == 0): dlogits as launch_topk_gate_bwd would write from dgate.
cudaError_t launch_combine_bwd(const int32_t* row, const int32_t* counts, const int32_t* offsets,
                               long long rows, int zero_fill, const float* gate, int s, int k,
                               int e, int m, int dtype, const void* dout, const void* y, void* dY,
                               float* dgate, int sparse, const DeviceInfo& di, cudaStream_t st,
                               const int32_t* rg_idx = nullptr, const float* rg_logits = nullptr,
                               int rg_renorm = 1, float* rg_dlogits = nullptr);

// --- per-virtual-rank send slots ------------------------------------------
// rank_slot[t,r] = token-order position of t among the tokens sending to r,
// -1 where token_in_rank[t,r] = 0.  [s,R] int32, one CTA per rank.
cudaError_t launch_rank_slots(const uint8_t* token_in_rank, int s, int R, int32_t* rank_slot,
                              cudaStream_t st);

// --- expert-parallel exchange: send map and gate gradients ---------------
// send_row [s,R], meta_idx / meta_gate [rows_sent,k] (see ep.cu).
cudaError_t launch_ep_pack(const int32_t* idx, const int32_t* row, const float* gate, const int32_t* rank_slot,
                           const int32_t* rank_counts, int s, int k, int e, int R, long long rows_sent,
                           int32_t* send_row, int32_t* meta_idx, float* meta_gate, int32_t* status,
                           const DeviceInfo& di, cudaStream_t st);
// dgate[t,j] = dgate_back[send_row[t, idx[t,j]/E], j] for kept routes, else 0.
cudaError_t launch_ep_unpack_dgate(const int32_t* idx, const int32_t* row, const int32_t* send_row,
                                   const float* dgate_back, int s, int k, int e, int R, long long rows_sent,
                                   float* dgate, const DeviceInfo& di, cudaStream_t st);

// --- expert-grouped GEMM on the tensor cores -----------------------------
// Y[r] = X[r] . W[x]^T over the 128-row blocks of each expert segment that a
// route owns.  K % 8 == 0 (>= 64), N % 8 == 0; a segment may start on any row.
cudaError_t launch_grouped_gemm(const int32_t* offsets, const int32_t* counts, int e, int rows, int K,
                                int N, const void* X, const void* W, void* Y, int32_t* status,
                                const DeviceInfo& di, cudaStream_t st);

// Fused dispatch + grouped GEMM: A rows gathered from the token rows x [s,K]
// through inv_row; same output as launch_grouped_gemm on the dispatched rows.
cudaError_t launch_dispatch_gemm(const int32_t* offsets, const int32_t* counts, const int32_t* inv_row,
                                 int e, int rows, int s, int K, int N, const void* x, const void* W,
                                 void* Y, int32_t* status, const DeviceInfo& di, cudaStream_t st);

}  // namespace moe
