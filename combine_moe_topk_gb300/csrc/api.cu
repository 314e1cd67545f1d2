// api.cu -- the C ABI of libmoe_gb300 (declared in include/moe_gb300.h):
// host-side validation, the layout handle and its stream-ordered memory,
// launch counters, and the calls into the kernel launchers.
//
// Validation runs entirely on the host and before the first CUDA call of an
// entry point, so a rejected call enqueues nothing (and works without a GPU).
#include <cuda_runtime.h>
#include <stdio.h>
#include <string.h>

#include <atomic>
#include <cmath>
#include <mutex>
#include <string>
#include <unordered_set>

#include "../../include/moe_gb300.h"
#include "internal.h"

struct moe_handle_s {
  int device;
  cudaStream_t stream;
  int s, e, k, capacity, R, rows;
  int priority, pad;
  int zero_fill;  // the dispatched buffer has rows no route owns
  void* blob;
  size_t blob_bytes;
  size_t clear_bytes;  // the blob's leading status word and rank counts
  moe::LayoutOut out;
  int32_t* rank_slot;  // [s,R] send slots, or NULL
  moe::LayoutPlan plan;
  int builds;          // layout builds enqueued so far (0: created, no layout yet)
  int absent;          // expert id -1 = an absent route
};

namespace {

thread_local std::string g_last_error;
std::atomic<uint64_t> g_launches[MOE_KERNEL_COUNT];
std::mutex g_mu;
std::unordered_set<const moe_handle_s*> g_live;  // handles not yet destroyed
int g_hold_tile = -1;                            // test hook, see moe_debug_hold_layout_tile
long long g_hold_timeout_ns = 0;

constexpr int kMaxDevices = 64;
constexpr int kMaxE = 256;
constexpr int kMaxK = 16;
constexpr int kMaxR = 64;
constexpr long long kDefaultTimeoutNs = 2000000000LL;  // bounded device waits: 2 s

moe_status fail(moe_status st, const std::string& why) {
  g_last_error = why;
  return st;
}

moe_status cuda_fail(cudaError_t err, const char* where) {
  g_last_error = std::string(where) + ": " + cudaGetErrorString(err);
  return err == cudaErrorMemoryAllocation ? MOE_ERR_OOM : MOE_ERR_CUDA;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// Host-only checks of a payload row: dtype and 16-byte row length.
moe_status check_payload(moe_dtype dt, int m, long long* row_bytes) {
  if (dt == MOE_F16) return fail(MOE_ERR_DTYPE, "fp16 activations are not supported; use bf16 or fp32");
  if (dt != MOE_F32 && dt != MOE_BF16) return fail(MOE_ERR_DTYPE, "unknown dtype");
  if (m < 1) return fail(MOE_ERR_INVALID_ARG, "m must be >= 1");
  const long long rb = (long long)m * (dt == MOE_F32 ? 4 : 2);
  if (rb % 16 != 0) return fail(MOE_ERR_INVALID_ARG, "a payload row (m * element size) must be a multiple of 16 bytes");
  *row_bytes = rb;
  return MOE_OK;
}

moe_status check_ptr(const void* p, const char* name, bool may_be_null = false) {
  if (!p) {
    if (may_be_null) return MOE_OK;
    return fail(MOE_ERR_INVALID_ARG, std::string(name) + " is NULL");
  }
  if (!aligned16(p)) return fail(MOE_ERR_INVALID_ARG, std::string(name) + " is not 16-byte aligned");
  return MOE_OK;
}

// Device residency: a pointer the kernels can dereference on `device`.
moe_status check_device_ptr(const void* p, const char* name, int device) {
  if (!p) return MOE_OK;
  cudaPointerAttributes a;
  cudaError_t err = cudaPointerGetAttributes(&a, p);
  if (err != cudaSuccess) {
    cudaGetLastError();
    return fail(MOE_ERR_INVALID_ARG, std::string(name) + ": not a CUDA pointer");
  }
  if (a.type == cudaMemoryTypeManaged) return MOE_OK;
  if (a.type != cudaMemoryTypeDevice)
    return fail(MOE_ERR_INVALID_ARG, std::string(name) + " is not device memory");
  if (a.device != device)
    return fail(MOE_ERR_INVALID_ARG, std::string(name) + " lives on another device");
  return MOE_OK;
}

#define MOE_TRY(expr)               \
  do {                              \
    moe_status _st = (expr);        \
    if (_st != MOE_OK) return _st;  \
  } while (0)

moe_status live_handle(moe_handle h) {
  if (!h) return fail(MOE_ERR_INVALID_ARG, "handle is NULL");
  std::lock_guard<std::mutex> lk(g_mu);
  if (!g_live.count(h)) return fail(MOE_ERR_HANDLE_MISMATCH, "handle is unknown or destroyed");
  return MOE_OK;
}

// A handle from moe_layout_create has no layout until its first build.
moe_status built_handle(moe_handle h) {
  MOE_TRY(live_handle(h));
  if (h->builds == 0) return fail(MOE_ERR_INVALID_ARG, "the handle has no layout yet (build it first)");
  return MOE_OK;
}

moe_status check_shape(moe_handle h, int s, int rows) {
  if (s != h->s)
    return fail(MOE_ERR_HANDLE_MISMATCH, "token count " + std::to_string(s) + " differs from the handle's " + std::to_string(h->s));
  if (rows != h->rows)
    return fail(MOE_ERR_HANDLE_MISMATCH, "row count " + std::to_string(rows) + " differs from the handle's " + std::to_string(h->rows));
  return MOE_OK;
}

moe_status current_device(int* dev) {
  cudaError_t err = cudaGetDevice(dev);
  if (err != cudaSuccess) return cuda_fail(err, "cudaGetDevice");
  if (*dev < 0 || *dev >= kMaxDevices) return fail(MOE_ERR_UNSUPPORTED, "device ordinal too large");
  return MOE_OK;
}

moe_status handle_device(moe_handle h) {
  int dev = 0;
  MOE_TRY(current_device(&dev));
  if (dev != h->device) return fail(MOE_ERR_HANDLE_MISMATCH, "the current device is not the handle's device");
  return MOE_OK;
}

// ---- per-device state --------------------------------------------------------

std::once_flag g_dev_once[kMaxDevices];
moe::DeviceInfo g_dev_info[kMaxDevices];
cudaMemPool_t g_pool[kMaxDevices];
cudaError_t g_dev_err[kMaxDevices];

void init_device(int dev) {
  moe::DeviceInfo& di = g_dev_info[dev];
  cudaError_t err = cudaDeviceGetAttribute(&di.sms, cudaDevAttrMultiProcessorCount, dev);
  if (err == cudaSuccess)
    err = cudaDeviceGetAttribute(&di.max_smem_optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev);
  if (err == cudaSuccess) {
    di.layout_blocks_per_sm = moe::layout_blocks_per_sm();
    di.gate_layout_blocks_per_sm = moe::gate_layout_blocks_per_sm();
  }
  if (err == cudaSuccess) {
    cudaMemPoolProps props = {};
    props.allocType = cudaMemAllocationTypePinned;
    props.location.type = cudaMemLocationTypeDevice;
    props.location.id = dev;
    err = cudaMemPoolCreate(&g_pool[dev], &props);
    if (err == cudaSuccess) {
      // keep freed blocks in the pool: handles are built and destroyed per step
      uint64_t keep = UINT64_MAX;
      err = cudaMemPoolSetAttribute(g_pool[dev], cudaMemPoolAttrReleaseThreshold, &keep);
    }
  }
  g_dev_err[dev] = err;
}

moe_status device_state(int dev, const moe::DeviceInfo** di) {
  std::call_once(g_dev_once[dev], init_device, dev);
  if (g_dev_err[dev] != cudaSuccess) return cuda_fail(g_dev_err[dev], "device initialisation");
  *di = &g_dev_info[dev];
  return MOE_OK;
}

size_t align_up(size_t v, size_t a) { return (v + a - 1) / a * a; }

}  // namespace

namespace moe {
const DeviceInfo& device_info(int device) { return g_dev_info[device]; }
}  // namespace moe

extern "C" {

const char* moe_status_string(moe_status st) {
  switch (st) {
    case MOE_OK: return "ok";
    case MOE_ERR_INVALID_ARG: return "invalid argument";
    case MOE_ERR_UNSUPPORTED: return "unsupported";
    case MOE_ERR_DTYPE: return "unsupported dtype (fp32 and bf16 only)";
    case MOE_ERR_HANDLE_MISMATCH: return "handle mismatch";
    case MOE_ERR_CUDA: return "CUDA error";
    case MOE_ERR_OOM: return "out of device memory";
    case MOE_ERR_TIMEOUT: return "device wait timed out";
    case MOE_ERR_NONFINITE: return "non-finite logit";
    case MOE_ERR_BAD_ROUTE: return "expert id out of range or repeated in a token";
  }
  return "unknown status";
}

const char* moe_last_error(void) { return g_last_error.c_str(); }

uint64_t moe_launch_count(int kernel_id) {
  if (kernel_id < 0 || kernel_id >= MOE_KERNEL_COUNT) return 0;
  return g_launches[kernel_id].load();
}

int moe_capacity(double capacity_factor, int s, int k, int e) {
  if (!(capacity_factor > 0.0) || !std::isfinite(capacity_factor) || s < 0 || k < 1 || e < 1) return 0;
  const double c = std::ceil(capacity_factor * (double)s * (double)k / (double)e);
  if (c > 2147483647.0) return 0;
  return (int)c;
}

moe_status moe_debug_hold_layout_tile(int tile, int timeout_ms) {
  if (timeout_ms < 1 || timeout_ms > 10000) return fail(MOE_ERR_INVALID_ARG, "timeout_ms must be in [1, 10000]");
  std::lock_guard<std::mutex> lk(g_mu);
  g_hold_tile = tile < 0 ? -1 : tile;
  g_hold_timeout_ns = (long long)timeout_ms * 1000000LL;
  return MOE_OK;
}

moe_status moe_topk_gate(const float* logits, int s, int e, int k, int renorm, int32_t* topk_idx,
                         float* topk_gate, int32_t* device_status, void* stream) {
  if (s < 0 || e < 1 || e > kMaxE || k < 1 || k > e || k > kMaxK)
    return fail(MOE_ERR_INVALID_ARG, "need s >= 0, 1 <= e <= 256, 1 <= k <= min(e, 16)");
  if ((long long)s * k > 2147483647LL) return fail(MOE_ERR_INVALID_ARG, "s*k must be < 2^31");
  if (renorm != 0 && renorm != 1) return fail(MOE_ERR_INVALID_ARG, "renorm must be 0 or 1");
  if (s == 0) return MOE_OK;
  MOE_TRY(check_ptr(logits, "logits"));
  MOE_TRY(check_ptr(topk_idx, "topk_idx"));
  MOE_TRY(check_ptr(topk_gate, "topk_gate"));
  if (device_status && (reinterpret_cast<uintptr_t>(device_status) & 3u))
    return fail(MOE_ERR_INVALID_ARG, "device_status is not 4-byte aligned");
  int dev = 0;
  MOE_TRY(current_device(&dev));
  MOE_TRY(check_device_ptr(logits, "logits", dev));
  MOE_TRY(check_device_ptr(topk_idx, "topk_idx", dev));
  MOE_TRY(check_device_ptr(topk_gate, "topk_gate", dev));
  MOE_TRY(check_device_ptr(device_status, "device_status", dev));
  const moe::DeviceInfo* di = nullptr;
  MOE_TRY(device_state(dev, &di));
  cudaError_t err = moe::launch_topk_gate(logits, s, e, k, renorm, topk_idx, topk_gate, device_status,
                                          *di, static_cast<cudaStream_t>(stream));
  if (err != cudaSuccess) return cuda_fail(err, "topk_gate launch");
  g_launches[MOE_KERNEL_TOPK_GATE]++;
  return MOE_OK;
}

moe_status moe_topk_gate_bwd(const float* logits, const int32_t* topk_idx, const float* topk_gate,
                             const float* dgate, int s, int e, int k, int renorm, float* dlogits,
                             void* stream) {
  if (s < 0 || e < 1 || e > kMaxE || k < 1 || k > e || k > kMaxK)
    return fail(MOE_ERR_INVALID_ARG, "need s >= 0, 1 <= e <= 256, 1 <= k <= min(e, 16)");
  if ((long long)s * e > 2147483647LL) return fail(MOE_ERR_INVALID_ARG, "s*e must be < 2^31");
  if (renorm != 0 && renorm != 1) return fail(MOE_ERR_INVALID_ARG, "renorm must be 0 or 1");
  if (s == 0) return MOE_OK;
  if (!renorm) MOE_TRY(check_ptr(logits, "logits"));
  MOE_TRY(check_ptr(topk_idx, "topk_idx"));
  MOE_TRY(check_ptr(topk_gate, "topk_gate"));
  MOE_TRY(check_ptr(dgate, "dgate"));
  MOE_TRY(check_ptr(dlogits, "dlogits"));
  int dev = 0;
  MOE_TRY(current_device(&dev));
  const void* ptrs[5] = {renorm ? nullptr : logits, topk_idx, topk_gate, dgate, dlogits};
  const char* names[5] = {"logits", "topk_idx", "topk_gate", "dgate", "dlogits"};
  for (int i = 0; i < 5; ++i) MOE_TRY(check_device_ptr(ptrs[i], names[i], dev));
  const moe::DeviceInfo* di = nullptr;
  MOE_TRY(device_state(dev, &di));
  cudaError_t err = moe::launch_topk_gate_bwd(renorm ? nullptr : logits, topk_idx, topk_gate, dgate, s, e,
                                              k, renorm, dlogits, *di, static_cast<cudaStream_t>(stream));
  if (err != cudaSuccess) return cuda_fail(err, "topk_gate_bwd launch");
  g_launches[MOE_KERNEL_TOPK_GATE_BWD]++;
  return MOE_OK;
}

namespace {

// Validates the sizes and options, allocates the handle's blob from the
// device's pool on `stream` and zeroes its leading part (status word, rank
// counts, look-back words).  No layout yet.
moe_status create_handle(int s, int e, int k, const moe_layout_options* options, void* stream,
                         moe_handle* out, const int32_t* topk_idx = nullptr) {
  if (!out) return fail(MOE_ERR_INVALID_ARG, "out is NULL");
  *out = nullptr;
  if (!options) return fail(MOE_ERR_INVALID_ARG, "options is NULL");
  const int capacity = options->capacity;
  const int R = options->num_virtual_ranks;
  const int priority = options->priority;
  const int pad = options->pad_multiple < 1 ? 1 : options->pad_multiple;
  if (priority != MOE_PRIORITY_TOKEN && priority != MOE_PRIORITY_KMAJOR)
    return fail(MOE_ERR_INVALID_ARG, "unknown priority");
  if (pad > 1 && capacity > 0) return fail(MOE_ERR_INVALID_ARG, "pad_multiple applies to the dropless layout only");
  if (pad > 65536) return fail(MOE_ERR_INVALID_ARG, "pad_multiple must be <= 65536");
  const int send_slots = options->send_slots;
  if (send_slots != 0 && send_slots != 1) return fail(MOE_ERR_INVALID_ARG, "send_slots must be 0 or 1");
  if (options->absent_routes != 0 && options->absent_routes != 1)
    return fail(MOE_ERR_INVALID_ARG, "absent_routes must be 0 or 1");
  if (send_slots && options->num_virtual_ranks <= 0)
    return fail(MOE_ERR_INVALID_ARG, "send_slots needs num_virtual_ranks > 0");
  // with absent routes a token may list more routes than there are experts
  // (at most e of them present)
  if (s < 0 || e < 1 || e > kMaxE || k < 1 || (k > e && !options->absent_routes) || k > kMaxK)
    return fail(MOE_ERR_INVALID_ARG, "need s >= 0, 1 <= e <= 256, 1 <= k <= min(e, 16)");
  if (capacity < 0) return fail(MOE_ERR_INVALID_ARG, "capacity must be >= 0 (0 = dropless)");
  if (R < 0 || R > kMaxR || (R > 0 && e % R != 0))
    return fail(MOE_ERR_INVALID_ARG, "num_virtual_ranks must be in [0, 64] and divide e");
  const long long routes = (long long)s * k;
  long long rows = capacity > 0 ? (long long)e * capacity : routes + (long long)e * (pad - 1);
  if (routes > 2147483647LL || rows > 2147483647LL)
    return fail(MOE_ERR_INVALID_ARG, "s*k and the row count must be < 2^31");
  if ((long long)s * e > 2147483647LL) return fail(MOE_ERR_INVALID_ARG, "s*e must be < 2^31");
  if (options->rows_bound != 0) {
    if (capacity > 0 || pad > 1) return fail(MOE_ERR_INVALID_ARG, "rows_bound applies to the unpadded dropless layout");
    if (options->rows_bound < 0 || options->rows_bound > routes)
      return fail(MOE_ERR_INVALID_ARG, "rows_bound must be in [0, s*k]");
    rows = options->rows_bound;
  }

  if (topk_idx && s > 0) MOE_TRY(check_ptr(topk_idx, "topk_idx"));

  int dev = 0;
  MOE_TRY(current_device(&dev));
  if (topk_idx && s > 0) MOE_TRY(check_device_ptr(topk_idx, "topk_idx", dev));
  const moe::DeviceInfo* di = nullptr;
  MOE_TRY(device_state(dev, &di));

  moe_handle_s* h = new moe_handle_s();
  h->device = dev;
  h->stream = static_cast<cudaStream_t>(stream);
  h->s = s;
  h->e = e;
  h->k = k;
  h->capacity = capacity;
  h->R = R;
  h->rows = (int)rows;
  h->priority = priority;
  h->pad = pad;
  h->zero_fill = capacity > 0 || pad > 1;
  h->builds = 0;
  h->absent = options->absent_routes != 0;
  // the scan runs over s*k one-route units in k-major order
  h->plan = moe::plan_layout(priority == MOE_PRIORITY_KMAJOR ? s * k : s, e, *di);

  // one blob: [zeroed: status, rank_counts, look-back words] then the rest
  const size_t A = 256;
  size_t off = 0;
  const size_t o_status = off; off = align_up(off + 4, A);
  const size_t o_rank = off;   off = align_up(off + 4 * (size_t)(R > 0 ? R : 1), A);
  h->clear_bytes = off;
  const size_t o_lb = off;     off = align_up(off + moe::lookback_bytes(h->plan, e), A);
  const size_t zero_bytes = off;
  const size_t o_idx = off;    off = align_up(off + 4 * (size_t)routes, A);
  const size_t o_loc = off;    off = align_up(off + 4 * (size_t)routes, A);
  const size_t o_row = off;    off = align_up(off + 4 * (size_t)routes, A);
  const size_t o_drop = off;   off = align_up(off + (size_t)routes, A);
  const size_t o_raw = off;    off = align_up(off + 4 * (size_t)e, A);
  const size_t o_cnt = off;    off = align_up(off + 4 * (size_t)e, A);
  const size_t o_off = off;    off = align_up(off + 4 * (size_t)(e + 1), A);
  const size_t o_tir = off;    off = align_up(off + (size_t)s * (R > 0 ? R : 0) + 1, A);
  const size_t o_inv = off;    off = align_up(off + 4 * (size_t)rows + 4, A);
  const size_t o_slot = off;   off = align_up(off + (send_slots ? 4 * (size_t)s * R : 0), A);
  h->blob_bytes = off;

  cudaError_t err = cudaMallocFromPoolAsync(&h->blob, h->blob_bytes, g_pool[dev], h->stream);
  if (err != cudaSuccess) {
    delete h;
    return cuda_fail(err, "handle allocation");
  }
  char* base = static_cast<char*>(h->blob);
  h->out.status = reinterpret_cast<int32_t*>(base + o_status);
  h->out.rank_counts = R > 0 ? reinterpret_cast<int32_t*>(base + o_rank) : nullptr;
  h->out.lookback = reinterpret_cast<unsigned*>(base + o_lb);
  h->out.idx = reinterpret_cast<int32_t*>(base + o_idx);
  h->out.loc = reinterpret_cast<int32_t*>(base + o_loc);
  h->out.row = reinterpret_cast<int32_t*>(base + o_row);
  h->out.drop = reinterpret_cast<uint8_t*>(base + o_drop);
  h->out.raw_counts = reinterpret_cast<int32_t*>(base + o_raw);
  h->out.counts = reinterpret_cast<int32_t*>(base + o_cnt);
  h->out.offsets = reinterpret_cast<int32_t*>(base + o_off);
  h->out.token_in_rank = R > 0 ? reinterpret_cast<uint8_t*>(base + o_tir) : nullptr;
  h->out.inv_row = reinterpret_cast<int32_t*>(base + o_inv);
  h->rank_slot = send_slots ? reinterpret_cast<int32_t*>(base + o_slot) : nullptr;

  err = cudaMemsetAsync(base, 0, zero_bytes, h->stream);
  if (err != cudaSuccess) {
    cudaFreeAsync(h->blob, h->stream);
    delete h;
    return cuda_fail(err, "handle zeroing");
  }
  {
    std::lock_guard<std::mutex> lk(g_mu);
    g_live.insert(h);
  }
  *out = h;
  return MOE_OK;
}

// Enqueues one build of h's layout on `stream`: from expert ids, or (logits
// != nullptr) with the top-k gate fused in, writing the ids and gates to
// gate_idx / gate_val.  Nothing here depends on how many builds came before
// (the kernel finds its look-back parity on the device and clears the status
// word and rank counts itself), so a CUDA graph may capture a build and
// replay it.
moe_status build_handle(moe_handle h, const int32_t* topk_idx, const float* logits, int renorm,
                        int32_t* gate_idx, float* gate_val, void* stream) {
  const cudaStream_t st = static_cast<cudaStream_t>(stream);
  moe::LayoutBuild build;
  build.clear_status = 1;
  build.absent_ok = h->absent;
  cudaError_t err = cudaSuccess;
  const moe::DeviceInfo* di = nullptr;
  MOE_TRY(device_state(h->device, &di));
  if (logits && !moe::layout_can_fuse_gate(h->plan, h->priority, h->e, *di)) {
    // the layout kernel cannot select in its first pass here: the gate
    // kernel first, then the layout on its ids (the status word cleared
    // before the gate reports into it)
    err = cudaMemsetAsync(h->blob, 0, h->clear_bytes, st);
    if (err == cudaSuccess)
      err = moe::launch_topk_gate(logits, h->s, h->e, h->k, renorm, gate_idx, gate_val, h->out.status, *di, st);
    if (err != cudaSuccess) return cuda_fail(err, "topk_gate launch");
    g_launches[MOE_KERNEL_TOPK_GATE]++;
    topk_idx = gate_idx;
    logits = nullptr;
    build.clear_status = 0;
  }
  if (logits) {
    build.logits = logits;
    build.renorm = renorm;
    build.gate_idx = gate_idx;
    build.gate_val = gate_val;
  }
  int hold = -1;
  long long timeout_ns = kDefaultTimeoutNs;
  {
    std::lock_guard<std::mutex> lk(g_mu);
    if (g_hold_tile >= 0 && g_hold_tile < h->plan.tiles) {
      hold = g_hold_tile;
      timeout_ns = g_hold_timeout_ns;
      g_hold_tile = -1;
    }
  }
  err = moe::launch_layout(topk_idx, h->s, h->e, h->k, h->capacity, h->R, h->priority, h->pad, h->rows, h->plan,
                           h->out, hold, timeout_ns, st, build);
  if (err != cudaSuccess) return cuda_fail(err, "layout launch");
  g_launches[logits ? MOE_KERNEL_GATE_LAYOUT : MOE_KERNEL_LAYOUT]++;
  h->builds++;
  h->stream = st;  // the handle's latest writer: its memory is freed on this stream
  if (h->rank_slot && h->s > 0) {
    err = moe::launch_rank_slots(h->out.token_in_rank, h->s, h->R, h->rank_slot, st);
    if (err != cudaSuccess) return cuda_fail(err, "rank_slots launch");
    g_launches[MOE_KERNEL_RANK_SLOTS]++;
  }
  return MOE_OK;
}

// Device-pointer checks of a build's inputs and outputs.
moe_status check_build_ptrs(moe_handle h, const int32_t* topk_idx, const float* logits, int32_t* gate_idx,
                            float* gate_val) {
  if (h->s == 0) return MOE_OK;
  MOE_TRY(handle_device(h));
  if (!logits) {
    MOE_TRY(check_ptr(topk_idx, "topk_idx"));
    return check_device_ptr(topk_idx, "topk_idx", h->device);
  }
  MOE_TRY(check_ptr(logits, "logits"));
  MOE_TRY(check_ptr(gate_idx, "topk_idx"));
  MOE_TRY(check_ptr(gate_val, "topk_gate"));
  MOE_TRY(check_device_ptr(logits, "logits", h->device));
  MOE_TRY(check_device_ptr(gate_idx, "topk_idx", h->device));
  return check_device_ptr(gate_val, "topk_gate", h->device);
}

// Removes a handle that failed its first build.
void discard_handle(moe_handle h) {
  {
    std::lock_guard<std::mutex> lk(g_mu);
    g_live.erase(h);
  }
  cudaFreeAsync(h->blob, h->stream);
  delete h;
}

}  // namespace

moe_status moe_dispatch_layout_ex(const int32_t* topk_idx, int s, int e, int k,
                                  const moe_layout_options* options, void* stream, moe_handle* out) {
  if (!out) return fail(MOE_ERR_INVALID_ARG, "out is NULL");
  *out = nullptr;
  if (s > 0 && !topk_idx) return fail(MOE_ERR_INVALID_ARG, "topk_idx is NULL");
  moe_handle h = nullptr;
  MOE_TRY(create_handle(s, e, k, options, stream, &h, topk_idx));
  const moe_status st = build_handle(h, topk_idx, nullptr, 1, nullptr, nullptr, stream);
  if (st != MOE_OK) {
    discard_handle(h);
    return st;
  }
  *out = h;
  return MOE_OK;
}

moe_status moe_layout_create(int s, int e, int k, const moe_layout_options* options, void* stream,
                             moe_handle* out) {
  return create_handle(s, e, k, options, stream, out);
}

moe_status moe_layout_rebuild(moe_handle h, const int32_t* topk_idx, void* stream) {
  MOE_TRY(live_handle(h));
  MOE_TRY(check_build_ptrs(h, topk_idx, nullptr, nullptr, nullptr));
  return build_handle(h, topk_idx, nullptr, 1, nullptr, nullptr, stream);
}

moe_status moe_topk_gate_layout(moe_handle h, const float* logits, int renorm, int32_t* topk_idx,
                                float* topk_gate, void* stream) {
  MOE_TRY(live_handle(h));
  if (renorm != 0 && renorm != 1) return fail(MOE_ERR_INVALID_ARG, "renorm must be 0 or 1");
  MOE_TRY(check_build_ptrs(h, nullptr, logits, topk_idx, topk_gate));
  return build_handle(h, nullptr, logits, renorm, topk_idx, topk_gate, stream);
}

moe_status moe_dispatch_layout(const int32_t* topk_idx, int s, int e, int k, int capacity,
                               int num_virtual_ranks, void* stream, moe_handle* out) {
  moe_layout_options opt;
  opt.capacity = capacity;
  opt.num_virtual_ranks = num_virtual_ranks;
  opt.priority = MOE_PRIORITY_TOKEN;
  opt.pad_multiple = 1;
  opt.send_slots = 0;
  opt.absent_routes = 0;
  opt.rows_bound = 0;
  return moe_dispatch_layout_ex(topk_idx, s, e, k, &opt, stream, out);
}

namespace {

// Sizes first; pointers only when there is work (a_rows rows of A, rows of Y).
moe_status check_gemm(moe_handle h, int rows, int K, int N, const void* A, const char* a_name, int a_rows,
                      const void* W, const void* Y) {
  if (rows != h->rows) return fail(MOE_ERR_HANDLE_MISMATCH, "row count differs from the handle's");
  if (K < 64 || K % 8 != 0) return fail(MOE_ERR_INVALID_ARG, "K must be a multiple of 8, at least 64");
  if (N < 8 || N % 8 != 0) return fail(MOE_ERR_INVALID_ARG, "N must be a positive multiple of 8");
  if ((long long)h->e * N > 2147483647LL) return fail(MOE_ERR_INVALID_ARG, "e * N must be < 2^31");
  if (rows == 0 || a_rows == 0) return MOE_OK;
  MOE_TRY(check_ptr(A, a_name));
  MOE_TRY(check_ptr(W, "W"));
  MOE_TRY(check_ptr(Y, "Y"));
  MOE_TRY(handle_device(h));
  MOE_TRY(check_device_ptr(A, a_name, h->device));
  MOE_TRY(check_device_ptr(W, "W", h->device));
  MOE_TRY(check_device_ptr(Y, "Y", h->device));
  return MOE_OK;
}

moe_status gemm_result(cudaError_t err, const char* where, int kernel) {
  if (err == cudaErrorInvalidValue) return fail(MOE_ERR_CUDA, "tensor-map encoding failed (driver entry point)");
  if (err != cudaSuccess) return cuda_fail(err, where);
  g_launches[kernel]++;
  return MOE_OK;
}

}  // namespace

moe_status moe_grouped_gemm(moe_handle h, int rows, int K, int N, const void* X, const void* W,
                            void* Y, void* stream) {
  MOE_TRY(built_handle(h));
  MOE_TRY(check_gemm(h, rows, K, N, X, "X", rows, W, Y));
  if (rows == 0) return MOE_OK;
  const moe::DeviceInfo* di = nullptr;
  MOE_TRY(device_state(h->device, &di));
  return gemm_result(moe::launch_grouped_gemm(h->out.offsets, h->out.counts, h->e, rows, K, N, X, W, Y,
                                              h->out.status, *di, static_cast<cudaStream_t>(stream)),
                     "grouped_gemm launch", MOE_KERNEL_GROUPED_GEMM);
}

moe_status moe_dispatch_grouped_gemm(moe_handle h, int s, int rows, int K, int N, const void* x,
                                     const void* W, void* Y, void* stream) {
  MOE_TRY(built_handle(h));
  MOE_TRY(check_shape(h, s, rows));
  MOE_TRY(check_gemm(h, rows, K, N, x, "x", s, W, Y));
  if (rows == 0 || s == 0) return MOE_OK;
  const moe::DeviceInfo* di = nullptr;
  MOE_TRY(device_state(h->device, &di));
  return gemm_result(moe::launch_dispatch_gemm(h->out.offsets, h->out.counts, h->out.inv_row, h->e, rows, s,
                                               K, N, x, W, Y, h->out.status, *di,
                                               static_cast<cudaStream_t>(stream)),
                     "dispatch_grouped_gemm launch", MOE_KERNEL_DISPATCH_GEMM);
}

namespace {

// An expert-parallel source handle and its send map: built, with send slots
// over 1..32 ranks, rows_sent in range, pointers on the handle's device.
moe_status check_ep(moe_handle h, int rows_sent, const void* send_row) {
  MOE_TRY(built_handle(h));
  if (h->R < 1 || h->R > 32) return fail(MOE_ERR_INVALID_ARG, "expert-parallel calls need 1 <= R <= 32 ranks");
  if (!h->rank_slot) return fail(MOE_ERR_INVALID_ARG, "the handle was built without send_slots");
  if (rows_sent < 0 || (long long)rows_sent > (long long)h->s * h->R)
    return fail(MOE_ERR_INVALID_ARG, "rows_sent must be in [0, s*R]");
  if (h->s > 0) {
    MOE_TRY(check_ptr(send_row, "send_row"));
    MOE_TRY(handle_device(h));
    MOE_TRY(check_device_ptr(send_row, "send_row", h->device));
  }
  return MOE_OK;
}

}  // namespace

moe_status moe_ep_pack(moe_handle h, const float* gate, int rows_sent, int32_t* send_row, int32_t* meta_idx,
                       float* meta_gate, void* stream) {
  MOE_TRY(check_ep(h, rows_sent, send_row));
  if ((long long)rows_sent * h->k > 2147483647LL) return fail(MOE_ERR_INVALID_ARG, "rows_sent*k must be < 2^31");
  if (h->s == 0) return MOE_OK;
  MOE_TRY(check_ptr(gate, "gate"));
  MOE_TRY(check_device_ptr(gate, "gate", h->device));
  if (rows_sent > 0) {
    MOE_TRY(check_ptr(meta_idx, "meta_idx"));
    MOE_TRY(check_ptr(meta_gate, "meta_gate"));
    MOE_TRY(check_device_ptr(meta_idx, "meta_idx", h->device));
    MOE_TRY(check_device_ptr(meta_gate, "meta_gate", h->device));
  }
  const moe::DeviceInfo* di = nullptr;
  MOE_TRY(device_state(h->device, &di));
  cudaError_t err = moe::launch_ep_pack(h->out.idx, h->out.row, gate, h->rank_slot, h->out.rank_counts, h->s, h->k,
                                        h->e, h->R, rows_sent, send_row, meta_idx, meta_gate, h->out.status, *di,
                                        static_cast<cudaStream_t>(stream));
  if (err != cudaSuccess) return cuda_fail(err, "ep_pack launch");
  g_launches[MOE_KERNEL_EP_PACK]++;
  return MOE_OK;
}

moe_status moe_ep_dispatch(moe_handle h, const int32_t* send_row, int rows_sent, int m, moe_dtype dtype,
                           const void* x, void* X_send, void* stream) {
  MOE_TRY(check_ep(h, rows_sent, send_row));
  long long rb = 0;
  MOE_TRY(check_payload(dtype, m, &rb));
  if (h->s == 0 || rows_sent == 0) return MOE_OK;
  MOE_TRY(check_ptr(x, "x"));
  MOE_TRY(check_ptr(X_send, "X_send"));
  MOE_TRY(check_device_ptr(x, "x", h->device));
  MOE_TRY(check_device_ptr(X_send, "X_send", h->device));
  const moe::DeviceInfo* di = nullptr;
  MOE_TRY(device_state(h->device, &di));
  cudaError_t err = moe::launch_dispatch(send_row, nullptr, nullptr, h->s, h->R, 1, rows_sent, 0, x, X_send, rb,
                                         h->out.status, *di, static_cast<cudaStream_t>(stream));
  if (err != cudaSuccess) return cuda_fail(err, "ep_dispatch launch");
  g_launches[MOE_KERNEL_EP_DISPATCH]++;
  return MOE_OK;
}

moe_status moe_ep_combine(moe_handle h, const int32_t* send_row, int rows_sent, int m, moe_dtype dtype,
                          const void* P, void* out, void* stream) {
  MOE_TRY(check_ep(h, rows_sent, send_row));
  long long rb = 0;
  MOE_TRY(check_payload(dtype, m, &rb));
  if (h->s == 0) return MOE_OK;
  if (rows_sent > 0) {
    MOE_TRY(check_ptr(P, "P"));
    MOE_TRY(check_device_ptr(P, "P", h->device));
  }
  MOE_TRY(check_ptr(out, "out"));
  MOE_TRY(check_device_ptr(out, "out", h->device));
  const moe::DeviceInfo* di = nullptr;
  MOE_TRY(device_state(h->device, &di));
  cudaError_t err = moe::launch_combine(send_row, nullptr, h->s, h->R, m, dtype == MOE_F32 ? 0 : 1, P, out, 1, *di,
                                        static_cast<cudaStream_t>(stream), rows_sent);
  if (err != cudaSuccess) return cuda_fail(err, "ep_combine launch");
  g_launches[MOE_KERNEL_EP_COMBINE]++;
  return MOE_OK;
}

moe_status moe_ep_unpack_dgate(moe_handle h, const int32_t* send_row, int rows_sent, const float* dgate_back,
                               float* dgate, void* stream) {
  MOE_TRY(check_ep(h, rows_sent, send_row));
  if (h->s == 0) return MOE_OK;
  if (rows_sent > 0) {
    MOE_TRY(check_ptr(dgate_back, "dgate_back"));
    MOE_TRY(check_device_ptr(dgate_back, "dgate_back", h->device));
  }
  MOE_TRY(check_ptr(dgate, "dgate"));
  MOE_TRY(check_device_ptr(dgate, "dgate", h->device));
  const moe::DeviceInfo* di = nullptr;
  MOE_TRY(device_state(h->device, &di));
  cudaError_t err = moe::launch_ep_unpack_dgate(h->out.idx, h->out.row, send_row, dgate_back, h->s, h->k, h->e, h->R,
                                                rows_sent, dgate, *di, static_cast<cudaStream_t>(stream));
  if (err != cudaSuccess) return cuda_fail(err, "ep_unpack_dgate launch");
  g_launches[MOE_KERNEL_EP_UNPACK]++;
  return MOE_OK;
}

moe_status moe_handle_info(moe_handle h, moe_layout_info* info) {
  MOE_TRY(live_handle(h));
  if (!info) return fail(MOE_ERR_INVALID_ARG, "info is NULL");
  info->s = h->s;
  info->e = h->e;
  info->k = h->k;
  info->capacity = h->capacity;
  info->R = h->R;
  info->rows = h->rows;
  info->device = h->device;
  info->priority = h->priority;
  info->pad_multiple = h->pad;
  info->idx = h->out.idx;
  info->loc = h->out.loc;
  info->row = h->out.row;
  info->drop = h->out.drop;
  info->raw_counts = h->out.raw_counts;
  info->counts = h->out.counts;
  info->offsets = h->out.offsets;
  info->token_in_rank = h->out.token_in_rank;
  info->rank_counts = h->out.rank_counts;
  info->status = h->out.status;
  info->inv_row = h->out.inv_row;
  info->rank_slot = h->rank_slot;
  return MOE_OK;
}

moe_status moe_handle_status(moe_handle h, void* stream, int32_t* device_status) {
  MOE_TRY(live_handle(h));
  if (!device_status) return fail(MOE_ERR_INVALID_ARG, "device_status is NULL");
  MOE_TRY(handle_device(h));
  cudaError_t err = cudaStreamSynchronize(static_cast<cudaStream_t>(stream));
  if (err == cudaSuccess) err = cudaStreamSynchronize(h->stream);
  if (err == cudaSuccess)
    err = cudaMemcpy(device_status, h->out.status, sizeof(int32_t), cudaMemcpyDeviceToHost);
  if (err != cudaSuccess) return cuda_fail(err, "reading the handle status");
  return MOE_OK;
}

moe_status moe_handle_destroy(moe_handle h) {
  if (!h) return fail(MOE_ERR_INVALID_ARG, "handle is NULL");
  {
    std::lock_guard<std::mutex> lk(g_mu);
    if (!g_live.erase(h)) return fail(MOE_ERR_HANDLE_MISMATCH, "handle is unknown or destroyed");
  }
  int prev = -1;
  cudaGetDevice(&prev);
  if (prev != h->device) cudaSetDevice(h->device);
  cudaError_t err = cudaFreeAsync(h->blob, h->stream);
  if (prev >= 0 && prev != h->device) cudaSetDevice(prev);
  delete h;
  if (err != cudaSuccess) return cuda_fail(err, "handle free");
  return MOE_OK;
}

moe_status moe_dispatch(moe_handle h, int s, int rows, int m, moe_dtype dtype, const void* x,
                        void* X, void* stream) {
  MOE_TRY(built_handle(h));
  MOE_TRY(check_shape(h, s, rows));
  long long rb = 0;
  MOE_TRY(check_payload(dtype, m, &rb));
  if (s > 0) MOE_TRY(check_ptr(x, "x"));
  if (rows > 0) MOE_TRY(check_ptr(X, "X"));
  MOE_TRY(handle_device(h));
  if (s > 0) MOE_TRY(check_device_ptr(x, "x", h->device));
  if (rows > 0) MOE_TRY(check_device_ptr(X, "X", h->device));
  if (rows == 0) return MOE_OK;
  const moe::DeviceInfo* di = nullptr;
  MOE_TRY(device_state(h->device, &di));
  cudaError_t err = moe::launch_dispatch(h->out.row, h->out.counts, h->out.offsets, s, h->k, h->e, h->rows,
                                         h->zero_fill, x, X, rb, h->out.status, *di,
                                         static_cast<cudaStream_t>(stream));
  if (err != cudaSuccess) return cuda_fail(err, "dispatch launch");
  g_launches[MOE_KERNEL_DISPATCH]++;
  return MOE_OK;
}

moe_status moe_combine(moe_handle h, int s, int rows, int m, moe_dtype dtype, const void* y,
                       const float* gate, void* out, void* stream) {
  MOE_TRY(built_handle(h));
  MOE_TRY(check_shape(h, s, rows));
  long long rb = 0;
  MOE_TRY(check_payload(dtype, m, &rb));
  if (s == 0) return MOE_OK;
  if (rows > 0) MOE_TRY(check_ptr(y, "y"));
  MOE_TRY(check_ptr(gate, "gate"));
  MOE_TRY(check_ptr(out, "out"));
  MOE_TRY(handle_device(h));
  if (rows > 0) MOE_TRY(check_device_ptr(y, "y", h->device));
  MOE_TRY(check_device_ptr(gate, "gate", h->device));
  MOE_TRY(check_device_ptr(out, "out", h->device));
  const moe::DeviceInfo* di = nullptr;
  MOE_TRY(device_state(h->device, &di));
  cudaError_t err = moe::launch_combine(h->out.row, gate, s, h->k, m, dtype == MOE_F32 ? 0 : 1, y, out, h->capacity > 0,
                                        *di, static_cast<cudaStream_t>(stream), h->rows);
  if (err != cudaSuccess) return cuda_fail(err, "combine launch");
  g_launches[MOE_KERNEL_COMBINE]++;
  return MOE_OK;
}

moe_status moe_combine_bwd(moe_handle h, int s, int rows, int m, moe_dtype dtype, const void* dout,
                           const float* gate, const void* y, void* dY, float* dgate, void* stream) {
  MOE_TRY(built_handle(h));
  MOE_TRY(check_shape(h, s, rows));
  long long rb = 0;
  MOE_TRY(check_payload(dtype, m, &rb));
  if (s == 0 && rows == 0) return MOE_OK;
  if (s > 0) {
    MOE_TRY(check_ptr(dout, "dout"));
    MOE_TRY(check_ptr(gate, "gate"));
    MOE_TRY(check_ptr(dgate, "dgate"));
  }
  if (rows > 0) {
    MOE_TRY(check_ptr(y, "y"));
    MOE_TRY(check_ptr(dY, "dY"));
  }
  MOE_TRY(handle_device(h));
  const void* ptrs[5] = {dout, gate, y, dY, dgate};
  const char* names[5] = {"dout", "gate", "y", "dY", "dgate"};
  for (int i = 0; i < 5; ++i) MOE_TRY(check_device_ptr(ptrs[i], names[i], h->device));
  const moe::DeviceInfo* di = nullptr;
  MOE_TRY(device_state(h->device, &di));
  cudaError_t err = moe::launch_combine_bwd(h->out.row, h->out.counts, h->out.offsets, h->rows,
                                            h->zero_fill, gate, s, h->k, h->e, m, dtype == MOE_F32 ? 0 : 1,
                                            dout, y, dY, dgate, h->capacity > 0, *di,
                                            static_cast<cudaStream_t>(stream));
  if (err != cudaSuccess) return cuda_fail(err, "combine_bwd launch");
  g_launches[MOE_KERNEL_COMBINE_BWD]++;
  return MOE_OK;
}

moe_status moe_combine_gate_bwd(moe_handle h, int s, int rows, int m, moe_dtype dtype,
                                const void* dout, const float* gate, const void* y,
                                const float* logits, int renorm, void* dY, float* dgate,
                                float* dlogits, void* stream) {
  MOE_TRY(built_handle(h));
  MOE_TRY(check_shape(h, s, rows));
  long long rb = 0;
  MOE_TRY(check_payload(dtype, m, &rb));
  if (renorm != 0 && renorm != 1) return fail(MOE_ERR_INVALID_ARG, "renorm must be 0 or 1");
  if ((long long)s * h->e > 2147483647LL) return fail(MOE_ERR_INVALID_ARG, "s*e must be < 2^31");
  if (s == 0 && rows == 0) return MOE_OK;
  if (s > 0) {
    MOE_TRY(check_ptr(dout, "dout"));
    MOE_TRY(check_ptr(gate, "gate"));
    MOE_TRY(check_ptr(dgate, "dgate"));
    MOE_TRY(check_ptr(dlogits, "dlogits"));
    if (!renorm) MOE_TRY(check_ptr(logits, "logits"));
  }
  if (rows > 0) {
    MOE_TRY(check_ptr(y, "y"));
    MOE_TRY(check_ptr(dY, "dY"));
  }
  MOE_TRY(handle_device(h));
  const void* ptrs[7] = {dout, gate, y, dY, dgate, dlogits, renorm ? nullptr : logits};
  const char* names[7] = {"dout", "gate", "y", "dY", "dgate", "dlogits", "logits"};
  for (int i = 0; i < 7; ++i) MOE_TRY(check_device_ptr(ptrs[i], names[i], h->device));
  const moe::DeviceInfo* di = nullptr;
  MOE_TRY(device_state(h->device, &di));
  cudaError_t err;
  if (s == 0) {  // nothing to route: only the zero rows of dY
    err = moe::launch_combine_bwd(h->out.row, h->out.counts, h->out.offsets, h->rows, h->zero_fill, gate,
                                  s, h->k, h->e, m, dtype == MOE_F32 ? 0 : 1, dout, y, dY, dgate,
                                  h->capacity > 0, *di, static_cast<cudaStream_t>(stream));
  } else {
    err = moe::launch_combine_bwd(h->out.row, h->out.counts, h->out.offsets, h->rows, h->zero_fill, gate,
                                  s, h->k, h->e, m, dtype == MOE_F32 ? 0 : 1, dout, y, dY, dgate,
                                  h->capacity > 0, *di, static_cast<cudaStream_t>(stream), h->out.idx,
                                  renorm ? nullptr : logits, renorm, dlogits);
  }
  if (err != cudaSuccess) return cuda_fail(err, "combine_gate_bwd launch");
  g_launches[s == 0 ? MOE_KERNEL_COMBINE_BWD : MOE_KERNEL_COMBINE_GATE_BWD]++;
  return MOE_OK;
}

moe_status moe_dispatch_bwd(moe_handle h, int s, int rows, int m, moe_dtype dtype, const void* dX,
                            void* dx, void* stream) {
  MOE_TRY(built_handle(h));
  MOE_TRY(check_shape(h, s, rows));
  long long rb = 0;
  MOE_TRY(check_payload(dtype, m, &rb));
  if (s == 0) return MOE_OK;
  if (rows > 0) MOE_TRY(check_ptr(dX, "dX"));
  MOE_TRY(check_ptr(dx, "dx"));
  MOE_TRY(handle_device(h));
  if (rows > 0) MOE_TRY(check_device_ptr(dX, "dX", h->device));
  MOE_TRY(check_device_ptr(dx, "dx", h->device));
  const moe::DeviceInfo* di = nullptr;
  MOE_TRY(device_state(h->device, &di));
  cudaError_t err = moe::launch_combine(h->out.row, nullptr, s, h->k, m, dtype == MOE_F32 ? 0 : 1, dX, dx, h->capacity > 0,
                                        *di, static_cast<cudaStream_t>(stream), h->rows);
  if (err != cudaSuccess) return cuda_fail(err, "dispatch_bwd launch");
  g_launches[MOE_KERNEL_DISPATCH_BWD]++;
  return MOE_OK;
}

moe_status moe_dispatch_layout_noalloc(const int32_t* topk_idx, int s, int e, int k, int capacity,
                                       int num_virtual_ranks, int32_t* idx_out, int32_t* loc,
                                       int32_t* row, uint8_t* drop, int32_t* raw_counts,
                                       int32_t* counts, int32_t* offsets, uint8_t* token_in_rank,
                                       int32_t* rank_counts, int32_t* device_status, void* stream) {
  const int R = num_virtual_ranks;
  if (s < 0 || e < 1 || e > kMaxE || k < 1 || k > e || k > kMaxK)
    return fail(MOE_ERR_INVALID_ARG, "need s >= 0, 1 <= e <= 256, 1 <= k <= min(e, 16)");
  if (capacity < 0) return fail(MOE_ERR_INVALID_ARG, "capacity must be >= 0 (0 = dropless)");
  if (R < 0 || R > kMaxR || (R > 0 && e % R != 0))
    return fail(MOE_ERR_INVALID_ARG, "num_virtual_ranks must be in [0, 64] and divide e");
  const long long routes = (long long)s * k;
  const long long rows = capacity > 0 ? (long long)e * capacity : routes;
  if (routes > 2147483647LL || rows > 2147483647LL)
    return fail(MOE_ERR_INVALID_ARG, "s*k and the row count must be < 2^31");
  void* per_route[5] = {const_cast<int32_t*>(topk_idx), idx_out, loc, row, drop};
  const char* route_names[5] = {"topk_idx", "idx_out", "loc", "row", "drop"};
  if (s > 0)
    for (int i = 0; i < 5; ++i) MOE_TRY(check_ptr(per_route[i], route_names[i]));
  MOE_TRY(check_ptr(raw_counts, "raw_counts"));
  MOE_TRY(check_ptr(counts, "counts"));
  MOE_TRY(check_ptr(offsets, "offsets"));
  if (R > 0) {
    MOE_TRY(check_ptr(rank_counts, "rank_counts"));
    if (s > 0) MOE_TRY(check_ptr(token_in_rank, "token_in_rank"));
  }
  if (device_status && (reinterpret_cast<uintptr_t>(device_status) & 3u))
    return fail(MOE_ERR_INVALID_ARG, "device_status is not 4-byte aligned");

  int dev = 0;
  MOE_TRY(current_device(&dev));
  const void* all[11] = {topk_idx, idx_out, loc, row, drop, raw_counts, counts, offsets,
                         R > 0 ? token_in_rank : nullptr, R > 0 ? rank_counts : nullptr,
                         device_status};
  const char* all_names[11] = {"topk_idx", "idx_out", "loc", "row", "drop", "raw_counts", "counts",
                               "offsets", "token_in_rank", "rank_counts", "device_status"};
  for (int i = 0; i < 11; ++i)
    if (i >= 5 || s > 0) MOE_TRY(check_device_ptr(all[i], all_names[i], dev));

  moe::LayoutOut out = {};
  out.idx = idx_out;
  out.loc = loc;
  out.row = row;
  out.drop = drop;
  out.raw_counts = raw_counts;
  out.counts = counts;
  out.offsets = offsets;
  out.token_in_rank = R > 0 ? token_in_rank : nullptr;
  out.rank_counts = R > 0 ? rank_counts : nullptr;
  out.status = device_status;
  int words = 0;
  cudaError_t err = moe::launch_layout_noalloc(topk_idx, s, e, k, capacity, R, out, &words,
                                               static_cast<cudaStream_t>(stream));
  if (err == cudaErrorInvalidValue && words > moe::noalloc_lookback_words())
    return fail(MOE_ERR_UNSUPPORTED,
                "the allocation-free layout needs " + std::to_string(words) +
                    " look-back words (tiles x experts) but holds " +
                    std::to_string(moe::noalloc_lookback_words()) + "; use moe_dispatch_layout");
  if (err != cudaSuccess) return cuda_fail(err, "allocation-free layout launch");
  g_launches[MOE_KERNEL_LAYOUT]++;
  return MOE_OK;
}

}  // extern "C"
