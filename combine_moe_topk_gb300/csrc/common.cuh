// common.cuh -- device helpers shared by the kernels of libmoe_gb300:
// status bits, bounded waits, 16-byte vector conversions, and the inline PTX
// for mbarriers and 1-D bulk (TMA) copies.  sm_103a only.
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <utility>

#include "../../include/moe_gb300.h"

namespace moe {

// ------------------------------------------------------------- status ------

__device__ __forceinline__ void raise_status(int32_t* status, int bits) {
  if (status) atomicOr(status, bits);
}

__device__ __forceinline__ uint64_t globaltimer_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

// ------------------------------------------- programmatic dependent launch --
// A kernel launched with programmatic stream serialisation may start while
// the previous kernel in the stream is still running; it must wait here
// before touching anything that kernel (or an earlier one) wrote.  A no-op
// when the kernel was launched without the attribute.
__device__ __forceinline__ void grid_dependency_wait() {
  asm volatile("griddepcontrol.wait;" ::: "memory");
}

// Let the next kernel in the stream begin its launch (it still waits for this
// grid to complete before reading its results).
__device__ __forceinline__ void grid_dependents_launch() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

// Where a kernel lets its dependent launch: 0 = programmatic launch off,
// 1 = as soon as the kernel may read its inputs, 2 = once its CTA's work is
// issued.
#ifndef MOE_PDL
#define MOE_PDL 2
#endif
__device__ __forceinline__ void pdl_trigger_early() {
  if (MOE_PDL == 1) grid_dependents_launch();
}
__device__ __forceinline__ void pdl_trigger_late() {
  if (MOE_PDL == 2) grid_dependents_launch();
}

// ------------------------------------------------------- row ownership -----
// Row r of a dispatched buffer whose expert segments are [offsets[x],
// offsets[x+1]) holds a route iff it lies in the first counts[x] rows of its
// segment (capacity slots past the count, per-expert padding and rows past
// offsets[e] hold none).  Binary search over the e + 1 offsets.
template <typename P>
__device__ __forceinline__ bool row_is_owned(long long r, const P* offsets, const P* counts, int e) {
  if (r >= (long long)offsets[e]) return false;
  int lo = 0, hi = e;  // offsets[lo] <= r < offsets[hi]
  while (hi - lo > 1) {
    const int mid = (lo + hi) >> 1;
    if ((long long)offsets[mid] <= r) lo = mid; else hi = mid;
  }
  return r - (long long)offsets[lo] < (long long)counts[lo];
}

// The per-expert segments (e + 1 offsets, e counts; e <= 256) staged in
// shared memory for a zero tail: one load per thread, all in flight at once,
// so the tail's ownership tests read shared memory instead of each running a
// chain of dependent global loads; read only after a block barrier.
struct SegmentStage {
  int offsets[257];
  int counts[256];
};

__device__ __forceinline__ void stage_segments(SegmentStage& st, const int32_t* offsets, const int32_t* counts,
                                               int e) {
  for (int x = threadIdx.x; x <= e; x += blockDim.x) {
    st.offsets[x] = __ldg(offsets + x);
    if (x < e) st.counts[x] = __ldg(counts + x);
  }
}

// ------------------------------------------------------ 16-byte vectors ----

template <typename T>
struct Vec;  // 16 bytes of T as floats

template <>
struct Vec<float> {
  static constexpr int N = 4;
  __device__ __forceinline__ static void to_float(const uint4& u, float* f) {
    f[0] = __uint_as_float(u.x);
    f[1] = __uint_as_float(u.y);
    f[2] = __uint_as_float(u.z);
    f[3] = __uint_as_float(u.w);
  }
  __device__ __forceinline__ static uint4 from_float(const float* f) {
    return make_uint4(__float_as_uint(f[0]), __float_as_uint(f[1]), __float_as_uint(f[2]),
                      __float_as_uint(f[3]));
  }
};

template <>
struct Vec<__nv_bfloat16> {
  static constexpr int N = 8;
  __device__ __forceinline__ static void to_float(const uint4& u, float* f) {
    const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      f[2 * i] = __uint_as_float(w[i] << 16);          // bf16 widening is a shift
      f[2 * i + 1] = __uint_as_float(w[i] & 0xffff0000u);
    }
  }
  __device__ __forceinline__ static uint4 from_float(const float* f) {
    uint32_t w[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      __nv_bfloat162 h = __floats2bfloat162_rn(f[2 * i], f[2 * i + 1]);  // nearest-even
      w[i] = *reinterpret_cast<uint32_t*>(&h);
    }
    return make_uint4(w[0], w[1], w[2], w[3]);
  }
};

// Streaming loads / stores: payload rows are touched once per kernel.
__device__ __forceinline__ uint4 ld_stream(const uint4* p) {
  uint4 v;
  asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "l"(p));
  return v;
}

__device__ __forceinline__ void st_stream(uint4* p, const uint4& v) {
  asm volatile("st.global.v4.u32 [%0], {%1,%2,%3,%4};" ::"l"(p), "r"(v.x), "r"(v.y), "r"(v.z),
               "r"(v.w)
               : "memory");
}

// ------------------------------------------------ mbarrier + bulk copies ---

__device__ __forceinline__ uint32_t smem_addr(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

// stage_segments with asynchronous 4-byte copies: issued at a kernel's start
// (after its programmatic-launch wait), so the loads travel while the kernel
// does its main work; segments_wait() (every thread) before reading them.
__device__ __forceinline__ void stage_segments_async(SegmentStage& st, const int32_t* offsets,
                                                     const int32_t* counts, int e) {
  for (int x = threadIdx.x; x <= e; x += blockDim.x) {
    asm volatile("cp.async.ca.shared.global [%0], [%1], 4;" ::"r"(smem_addr(&st.offsets[x])), "l"(offsets + x)
                 : "memory");
    if (x < e)
      asm volatile("cp.async.ca.shared.global [%0], [%1], 4;" ::"r"(smem_addr(&st.counts[x])), "l"(counts + x)
                   : "memory");
  }
}

__device__ __forceinline__ void segments_wait() {
  asm volatile("cp.async.wait_all;" ::: "memory");
  __syncthreads();
}

__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_addr(bar)), "r"(count)
               : "memory");
}

// Make mbarrier initialisation and generic-proxy shared-memory writes
// visible to the async proxy (the bulk-copy engine).
__device__ __forceinline__ void fence_barrier_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void fence_proxy_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_addr(bar)),
               "r"(bytes)
               : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(smem_addr(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}

// Bounded wait on an mbarrier phase.  Returns false if `deadline_ns` (on
// the global timer) passes first; the caller then records MOE_DEV_TIMEOUT.
__device__ __forceinline__ bool mbar_wait_bounded(uint64_t* bar, uint32_t parity,
                                                  uint64_t deadline_ns) {
  if (mbar_try_wait(bar, parity)) return true;
  for (uint32_t it = 0;; ++it) {
    if (mbar_try_wait(bar, parity)) return true;
    if ((it & 63) == 63 && globaltimer_ns() > deadline_ns) return false;
  }
}

// 1-D bulk copy global -> shared, completion counted on `bar` (bytes).
// Non-multicast; the destination is this CTA's own shared memory.
__device__ __forceinline__ void bulk_g2s(void* smem_dst, const void* gmem_src, uint32_t bytes,
                                         uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
          smem_addr(smem_dst)),
      "l"(gmem_src), "r"(bytes), "r"(smem_addr(bar))
      : "memory");
}

// 1-D bulk copy shared -> global, tracked by this thread's bulk async-group.
__device__ __forceinline__ void bulk_s2g(void* gmem_dst, const void* smem_src, uint32_t bytes) {
  asm volatile("cp.async.bulk.global.shared::cta.bulk_group [%0], [%1], %2;" ::"l"(gmem_dst),
               "r"(smem_addr(smem_src)), "r"(bytes)
               : "memory");
}

__device__ __forceinline__ void bulk_commit() {
  asm volatile("cp.async.bulk.commit_group;" ::: "memory");
}

// Wait until at most N of this thread's bulk groups still read shared memory.
template <int N>
__device__ __forceinline__ void bulk_wait_read() {
  asm volatile("cp.async.bulk.wait_group.read %0;" ::"n"(N) : "memory");
}

// Wait until all of this thread's bulk groups have completed.
__device__ __forceinline__ void bulk_wait_all() {
  asm volatile("cp.async.bulk.wait_group 0;" ::: "memory");
}

// Launch on `st` with programmatic stream serialisation: the kernel may begin
// while the previous kernel in the stream drains; it calls
// grid_dependency_wait() before reading anything that kernel wrote.
// Bit mask of the launches that use programmatic serialisation (bit i =
// kernel id i of moe_launch_count: gate 0, layout 1, dispatch 2, combine
// backward 4, dispatch backward 5, gate backward 6, combine + gate backward
// 10, the expert-parallel pack 12 and gate-gradient unpack 13).  The combine (3) is left out: its CTAs parked early on the SMs
// slowed the dispatch they follow, by 6-13 % of a step on every workload
// measured.
#ifndef MOE_PDL_MASK
#define MOE_PDL_MASK 0x3477
#endif

template <typename... KArgs, typename... Args>
cudaError_t launch_pdl(int kernel_id, void (*kern)(KArgs...), dim3 grid, dim3 block, size_t smem,
                       cudaStream_t st, Args&&... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = (MOE_PDL != 0 && ((MOE_PDL_MASK >> kernel_id) & 1)) ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, kern, std::forward<Args>(args)...);
}

}  // namespace moe
