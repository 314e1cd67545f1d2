// layout.cu -- the dispatch layout: per-expert counts, token-order slots,
// capacity drops or dropless grouped rows, and per-virtual-rank dedup counts,
// in one cooperative kernel.
//
// DeepSpeed #8195 "MoE dispatch: fix silent Tutel + TP corruption, speed up
// native and Tutel paths", changes 1 and 3: each route's slot inside its
// expert is the running count of earlier tokens sent to that expert
// (location = cumulative sum - 1, in token order), and routes past the
// capacity are dropped.  DeepSpeed #8213 "Add an opt-in DeepEP transport for
// the AutoEP expert all-to-all", description: a token is sent once per
// destination rank, so the dedup counts count tokens, not routes.
// Automodel #3684 "perf(moe): reuse the DeepEP dispatch layout on
// activation-checkpoint recompute": the layout must be reproducible, which
// rules out any result that depends on the order atomics arrive in.
//
// Structure.  Tile b (one CTA, 256 threads) owns a contiguous token range,
// processed as sub-tiles of 256 tokens (thread = token).
//   A. histogram: per-expert route count of the tile in shared memory
//      (integer atomics: the total does not depend on their order);
//   B. decoupled look-back over tiles, one thread per expert: publish the
//      tile aggregate, walk back to the nearest inclusive prefix, publish
//      the tile's inclusive prefix.  Flag and value share one 64-bit word.
//      The last tile's inclusive prefixes are the global expert totals;
//      dropless mode waits for them to form the row offsets;
//   C. slots: per sub-tile, each warp builds a 32-bit token mask per expert
//      (atomicOr: order-free), so a route's rank among the warp's tokens is
//      popc(mask & lanes-below); warps are scanned in order per expert.
// All waits are bounded on the global timer; when one runs out the kernel
// records MOE_DEV_TIMEOUT and carries on with what it has (no hang, no trap).
// All tiles are co-resident (cooperative launch), which is what makes the
// wait for the last tile safe.
#include <mutex>

#include "common.cuh"
#include "internal.h"

namespace moe {

namespace {

constexpr int kThreads = 256;  // also the sub-tile size in tokens
constexpr int kWarps = kThreads / 32;
constexpr int kMaxE = 256;
constexpr int kMaxK = 16;
constexpr int kMaxR = 64;

constexpr unsigned long long kFlagAgg = 1ull << 32;
constexpr unsigned long long kFlagPrefix = 2ull << 32;

struct Params {
  const int32_t* topk_idx;
  int s, e, k, capacity, R;
  int tiles, subtiles_per_tile;
  LayoutOut out;
  int hold_tile;
  long long timeout_ns;
};

// Load token t's k expert ids and mark which routes are valid: in range and
// not a repeat of an earlier route of the same token.
__device__ __forceinline__ unsigned load_routes(const Params& p, int t, int* xs) {
  unsigned valid = 0;
#pragma unroll
  for (int j = 0; j < kMaxK; ++j) {
    if (j < p.k) {
      const int x = __ldg(p.topk_idx + (size_t)t * p.k + j);
      xs[j] = x;
      bool ok = x >= 0 && x < p.e;
#pragma unroll
      for (int jj = 0; jj < j; ++jj)
        if (xs[jj] == x) ok = false;
      if (ok) valid |= 1u << j;
    }
  }
  return valid;
}

// Spin (bounded) until the look-back word carries a flag (any flag, or the
// inclusive-prefix flag when `want_prefix`).  Returns the word, or 0 with
// *timed_out set once the deadline has passed; after a time-out every later
// wait of this thread returns at once.
__device__ __forceinline__ unsigned long long wait_word(const unsigned long long* w,
                                                        bool want_prefix, uint64_t deadline,
                                                        bool* timed_out) {
  if (*timed_out) return 0;
  unsigned long long v = ld_relaxed_u64(w);
  for (uint32_t it = 0;; ++it) {
    const unsigned long long flag = v & ~0xffffffffull;
    if (want_prefix ? flag == kFlagPrefix : flag != 0) return v;
    __nanosleep(64);
    if ((it & 15) == 15 && globaltimer_ns() > deadline) {
      *timed_out = true;
      return 0;
    }
    v = ld_relaxed_u64(w);
  }
}

__global__ void __launch_bounds__(kThreads) layout_kernel(const Params p) {
  __shared__ int s_agg[kMaxE];       // tile aggregate per expert
  __shared__ int s_run[kMaxE];       // running slot base per expert
  __shared__ int s_off[kMaxE + 1];   // dropless row offsets
  __shared__ unsigned s_mask[kWarps][kMaxE];
  __shared__ int s_wbase[kWarps][kMaxE];
  __shared__ int s_rank[kMaxR];
  __shared__ int s_bad;
  __shared__ int s_timeout;

  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int tile = blockIdx.x;
  const int nsub = (p.s + kThreads - 1) / kThreads;
  const int sub0 = tile * p.subtiles_per_tile;
  const int sub1 = min(nsub, sub0 + p.subtiles_per_tile);
  const uint64_t deadline = globaltimer_ns() + (uint64_t)p.timeout_ns;

  for (int x = tid; x < kMaxE; x += kThreads) s_agg[x] = 0;
  if (tid < kMaxR) s_rank[tid] = 0;
  if (tid == 0) {
    s_bad = 0;
    s_timeout = 0;
  }
  __syncthreads();

  // ---- A: histogram of the tile, and the handle's copy of the ids --------
  int bad = 0;
  for (int sb = sub0; sb < sub1; ++sb) {
    const int t = sb * kThreads + tid;
    if (t < p.s) {
      int xs[kMaxK];
      const unsigned valid = load_routes(p, t, xs);
#pragma unroll
      for (int j = 0; j < kMaxK; ++j) {
        if (j < p.k) {
          p.out.idx[(size_t)t * p.k + j] = xs[j];
          if ((valid >> j) & 1u)
            atomicAdd(&s_agg[xs[j]], 1);
          else
            bad = 1;
        }
      }
    }
  }
  if (bad) s_bad = 1;
  __syncthreads();

  // ---- B: decoupled look-back over tiles, one thread per expert ----------
  bool timed_out = false;
  for (int x = tid; x < p.e; x += kThreads) {
    const int agg = s_agg[x];
    unsigned long long* col = p.out.lookback + x;  // word of tile b is col[b * e]
    const bool publish = tile != p.hold_tile;
    if (publish)
      st_relaxed_u64(col + (size_t)tile * p.e,
                     (tile == 0 ? kFlagPrefix : kFlagAgg) | (unsigned)agg);
    int excl = 0;
    for (int b = tile - 1; b >= 0; --b) {
      const unsigned long long w = wait_word(col + (size_t)b * p.e, false, deadline, &timed_out);
      if (timed_out) break;
      excl += (int)(unsigned)w;
      if ((w & ~0xffffffffull) == kFlagPrefix) break;
    }
    if (publish && tile > 0)
      st_relaxed_u64(col + (size_t)tile * p.e, kFlagPrefix | (unsigned)(excl + agg));
    s_run[x] = excl;

    // global totals = inclusive prefix of the last tile (dropless rows need
    // them in every tile; capacity mode only in the last tile, which has them)
    int total = excl + agg;
    if (p.capacity == 0 && tile != p.tiles - 1) {
      const unsigned long long w =
          wait_word(col + (size_t)(p.tiles - 1) * p.e, true, deadline, &timed_out);
      total = (int)(unsigned)w;
    }
    s_off[x] = total;  // holds totals until the scan below
  }
  if (timed_out) s_timeout = 1;
  __syncthreads();

  // totals -> counts, offsets (every tile in dropless mode; the last tile
  // alone also writes them to the handle)
  const bool last = tile == p.tiles - 1;
  if (p.capacity == 0 || last) {
    if (warp == 0) {
      // exclusive scan of e <= 256 counts: 8 per lane, then a warp scan
      int v[8];
      int sum = 0;
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        const int x = lane * 8 + i;
        int c = x < p.e ? s_off[x] : 0;
        if (p.capacity > 0) c = min(c, p.capacity);
        v[i] = c;
        sum += c;
      }
      int incl = sum;
#pragma unroll
      for (int off = 1; off < 32; off <<= 1) {
        const int o = __shfl_up_sync(0xffffffffu, incl, off);
        if (lane >= off) incl += o;
      }
      int run = incl - sum;
      int raw[8];
#pragma unroll
      for (int i = 0; i < 8; ++i) raw[i] = (lane * 8 + i) < p.e ? s_off[lane * 8 + i] : 0;
      __syncwarp();
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        const int x = lane * 8 + i;
        if (x < p.e) {
          const int off = p.capacity > 0 ? x * p.capacity : run;
          s_off[x] = off;
          if (last) {
            p.out.raw_counts[x] = raw[i];
            p.out.counts[x] = v[i];
            p.out.offsets[x] = off;
          }
        }
        run += v[i];
      }
      if (lane == 31) {
        const int end = p.capacity > 0 ? p.e * p.capacity : run;
        s_off[p.e] = end;
        if (last) p.out.offsets[p.e] = end;
      }
    }
    __syncthreads();
  }

  // ---- C: token-order slots, rows, drops, dedup ----------------------------
  const int per_rank = p.R > 0 ? p.e / p.R : 1;
  for (int sb = sub0; sb < sub1; ++sb) {
    for (int i = tid; i < kWarps * kMaxE; i += kThreads) (&s_mask[0][0])[i] = 0u;
    __syncthreads();
    const int t = sb * kThreads + tid;
    int xs[kMaxK];
    unsigned valid = 0;
    if (t < p.s) {
      valid = load_routes(p, t, xs);
#pragma unroll
      for (int j = 0; j < kMaxK; ++j)
        if ((valid >> j) & 1u) atomicOr(&s_mask[warp][xs[j]], 1u << lane);
    }
    __syncthreads();
    for (int x = tid; x < p.e; x += kThreads) {
      int run = s_run[x];
#pragma unroll
      for (int w = 0; w < kWarps; ++w) {
        s_wbase[w][x] = run;
        run += __popc(s_mask[w][x]);
      }
      s_run[x] = run;
    }
    __syncthreads();
    if (t < p.s) {
      const unsigned below = (1u << lane) - 1u;
      unsigned long long ranks = 0;
#pragma unroll
      for (int j = 0; j < kMaxK; ++j) {
        if (j < p.k) {
          const size_t q = (size_t)t * p.k + j;
          int loc = -1, row = -1;
          uint8_t drop = 1;
          if ((valid >> j) & 1u) {
            const int x = xs[j];
            loc = s_wbase[warp][x] + __popc(s_mask[warp][x] & below);
            if (p.capacity > 0) {
              drop = loc >= p.capacity;
              row = drop ? -1 : x * p.capacity + loc;
            } else {
              drop = 0;
              row = s_off[x] + loc;
            }
            if (!drop) ranks |= 1ull << (x / per_rank);
          }
          p.out.loc[q] = loc;
          p.out.row[q] = row;
          p.out.drop[q] = drop;
        }
      }
      if (p.R > 0) {
        uint8_t* tir = p.out.token_in_rank + (size_t)t * p.R;
        for (int r = 0; r < p.R; ++r) tir[r] = (uint8_t)((ranks >> r) & 1ull);
        while (ranks) {
          const int r = __ffsll((long long)ranks) - 1;
          ranks &= ranks - 1;
          atomicAdd(&s_rank[r], 1);
        }
      }
    }
    __syncthreads();
  }

  if (p.R > 0 && tid < p.R && s_rank[tid]) atomicAdd(&p.out.rank_counts[tid], s_rank[tid]);
  if (tid == 0) {
    int bits = 0;
    if (s_bad) bits |= MOE_DEV_BAD_ROUTE;
    if (s_timeout) bits |= MOE_DEV_TIMEOUT;
    if (bits) raise_status(p.out.status, bits);
  }
}

}  // namespace

LayoutPlan plan_layout(int s, const DeviceInfo& di) {
  LayoutPlan plan;
  const int nsub = s > 0 ? (s + kThreads - 1) / kThreads : 1;
  const int max_tiles = di.sms * (di.layout_blocks_per_sm > 0 ? di.layout_blocks_per_sm : 1);
  plan.subtiles_per_tile = (nsub + max_tiles - 1) / max_tiles;
  if (plan.subtiles_per_tile < 1) plan.subtiles_per_tile = 1;
  plan.tiles = (nsub + plan.subtiles_per_tile - 1) / plan.subtiles_per_tile;
  if (plan.tiles < 1) plan.tiles = 1;
  return plan;
}

int layout_blocks_per_sm() {
  int n = 0;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, layout_kernel, kThreads, 0) != cudaSuccess)
    return 0;
  return n;
}

cudaError_t launch_layout(const int32_t* topk_idx, int s, int e, int k, int capacity, int R,
                          const LayoutPlan& plan, const LayoutOut& out, int hold_tile,
                          long long timeout_ns, cudaStream_t st) {
  Params p;
  p.topk_idx = topk_idx;
  p.s = s;
  p.e = e;
  p.k = k;
  p.capacity = capacity;
  p.R = R;
  p.tiles = plan.tiles;
  p.subtiles_per_tile = plan.subtiles_per_tile;
  p.out = out;
  p.hold_tile = hold_tile;
  p.timeout_ns = timeout_ns;

  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(plan.tiles);
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = 0;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeCooperative;
  attr[0].val.cooperative = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, layout_kernel, p);
}

}  // namespace moe

// ---------------------------------------------------------------------------
// Allocation-free variant of the layout launch.
//
// For callers that cannot allocate device memory at the point they build a
// layout: code running inside a CUDA-graph-captured region where a pool
// allocation is not wanted, allocators that must not be re-entered (an
// allocator's own hook or a custom memory manager), or embedded runtimes
// that hand out only fixed buffers.  The caller passes every input and
// output; the kernel's only scratch -- the look-back words -- lives in the
// file-scope array below, which every GPU that loads this library holds
// until the process exits.
//
// The array is shared by every call on a device and keeps the last call's
// contents, so each call clears the words it uses first; calls whose
// kernels overlap on the GPU (different streams without ordering) race on it.
// ---------------------------------------------------------------------------
namespace moe {

constexpr int kNoAllocLookbackWords = 65536;  // 512 KB: tiles * e must fit

static __device__ __align__(256) unsigned long long g_noalloc_lookback[kNoAllocLookbackWords];

namespace {

struct NoAllocSetup {
  std::once_flag once;
  cudaError_t err = cudaSuccess;
  unsigned long long* scratch = nullptr;  // device address of g_noalloc_lookback
  DeviceInfo info;
};
NoAllocSetup g_noalloc[64];

// Once per device, with that device current: resolve the scratch array's
// device address (its host-side name is only a stand-in) and the sizes the
// tile plan needs.  Allocates nothing.
void noalloc_setup(int dev) {
  NoAllocSetup& st = g_noalloc[dev];
  void* ptr = nullptr;
  st.err = cudaGetSymbolAddress(&ptr, g_noalloc_lookback);
  if (st.err != cudaSuccess) return;
  st.scratch = static_cast<unsigned long long*>(ptr);
  st.err = cudaDeviceGetAttribute(&st.info.sms, cudaDevAttrMultiProcessorCount, dev);
  if (st.err != cudaSuccess) return;
  st.err = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&st.info.layout_blocks_per_sm, layout_kernel,
                                                         kThreads, 0);
}

}  // namespace

int noalloc_lookback_words() { return kNoAllocLookbackWords; }

cudaError_t launch_layout_noalloc(const int32_t* topk_idx, int s, int e, int k, int capacity, int R,
                                  const LayoutOut& out_in, int* words_needed, cudaStream_t st) {
  int dev = 0;
  cudaError_t err = cudaGetDevice(&dev);
  if (err != cudaSuccess) return err;
  if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  std::call_once(g_noalloc[dev].once, noalloc_setup, dev);
  const NoAllocSetup& setup = g_noalloc[dev];
  if (setup.err != cudaSuccess) return setup.err;

  const LayoutPlan plan = plan_layout(s, setup.info);
  const long long words = (long long)plan.tiles * e;
  *words_needed = (int)(words > 0x7fffffffLL ? 0x7fffffffLL : words);
  if (words > kNoAllocLookbackWords) return cudaErrorInvalidValue;  // caller reports the limit

  LayoutOut out = out_in;
  out.lookback = setup.scratch;
  err = cudaMemsetAsync(setup.scratch, 0, (size_t)words * sizeof(unsigned long long), st);
  if (err == cudaSuccess && R > 0)
    err = cudaMemsetAsync(out.rank_counts, 0, (size_t)R * sizeof(int32_t), st);
  if (err != cudaSuccess) return err;
  return launch_layout(topk_idx, s, e, k, capacity, R, plan, out, -1, 2000000000LL, st);
}

}  // namespace moe
