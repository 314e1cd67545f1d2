// grouped_gemm.cu -- the expert-grouped GEMM that consumes the dispatched
// rows, on the 5th-generation tensor cores (tcgen05, TMEM accumulators,
// TMA tile loads), and its fused form that gathers the token rows itself.
//
// DeepSpeed #8213 "Add an opt-in DeepEP transport for the AutoEP expert
// all-to-all", description: the dispatch groups arrivals by expert for the
// grouped GEMM, whose groups are bounded by offsets = cumsum(counts).
// Automodel #3684 "perf(moe): reuse the DeepEP dispatch layout on
// activation-checkpoint recompute": each expert's rows may be padded to a
// multiple (pad_multiple); nothing here needs it.
//
// Y[r] = A[r] . W[x]^T for every row r that a kept route to expert x owns,
// r in [offsets[x], offsets[x] + counts[x]).  A[r] is the dispatched row
// X[r] (moe_grouped_gemm) or the token row x[inv_row[r]] (fused dispatch:
// the dispatched buffer is never written or read).  bf16 operands,
// row-major, K contiguous; the accumulation is fp32 in TMEM.  Work units are row blocks
// of one expert's segment (256 rows on SM pairs, 128 on single SMs; the
// first at offsets[x], so a segment may start on any row) times
// 256-column tiles of N.
//
// Both forms run on pairs of SMs (grouped_gemm_pair_kernel, below): a
// cluster of two CTAs computes a 256-row block x 256 columns with
// tcgen05.mma.cta_group::2, each SM staging only its half of A and of B
// (two 64-wide K blocks per stage of a 3-stage ring).
// In the fused form the second CTA's gathered rows reach the MMA issuer
// through a 16-byte shared-to-shared bulk copy that counts on the first
// CTA's barrier: a per-K-block arrival with cluster-scope release instead
// held the paired fused GEMM to 0.56 PFLOP/s.  A TMA tile::gather4 of four
// rows per request was tried first for the fused form's A: correct, but at
// 33 copy requests per K-block it held the GEMM to a third of the tensor
// rate.  (A one-SM form with 128-row blocks came before the pairs and was
// measured 2-12 % slower on every shape; it is gone.  Short expert segments
// waste the tail of a 256-row block, but a 128-row block wastes the same
// tail rows, and where segments are short -- many experts, few rows each --
// streaming each expert's weights once bounds the GEMM anyway.)
// Every mbarrier wait is bounded on the global timer; a time-out records
// MOE_DEV_TIMEOUT and the roles wind down to the TMEM release.
#include <cuda.h>
#include <cudaTypedefs.h>

#include "common.cuh"
#include "internal.h"

namespace moe {

namespace {

constexpr int BM = 128, BN = 256, BK = 64;
constexpr int kTmemCols = 2 * BN;     // two fp32 accumulators of 128 lanes x 256 columns
constexpr int kThreads = 256;        // tile-fed form
// Warps gathering the fused form's A rows: 8 (16 rows each) measured 1-4 %
// faster than 4 and 3 % faster than 16 (fewer registers per thread at 768
// threads); 2 were 20-30 % slower.
#ifndef MOE_GEMM_GATHER_WARPS
#define MOE_GEMM_GATHER_WARPS 8
#endif
constexpr int kGatherThreads = kThreads + 32 * MOE_GEMM_GATHER_WARPS;  // fused form: + warps gathering A
constexpr int kGatherRows = BM / MOE_GEMM_GATHER_WARPS;  // A rows per gathering warp
static_assert(kGatherRows % 4 == 0 && kGatherRows >= 4, "a gathering warp copies 4 rows per instruction");
constexpr int kMaxE = 256;
// epilogue staging: per epilogue warp 32 rows x 64 bf16 columns, rows padded
// to 144 bytes (conflict-free 16-byte writes by row and reads by column)
constexpr int kStageRowBytes = 64 * 2 + 16;
constexpr int kEpiWarpBytes = 32 * kStageRowBytes;
constexpr int kEpiBytes = 4 * kEpiWarpBytes;

struct GemmParams {
  const __nv_bfloat16* x;  // gather mode: token rows [s, K]
  const int32_t* offsets;
  const int32_t* counts;
  const int32_t* inv_row;  // gather mode: token of each owned row
  int e, rows, K, N;
  int s;                   // gather mode: token rows of x
  __nv_bfloat16* Y;
  int32_t* status;
  long long timeout_ns;
};

// Shared-memory matrix descriptor: K-major, 128-byte swizzle (as TMA writes
// it), 8-row groups 1024 bytes apart.  The tile base is 1024-byte aligned.
__device__ __forceinline__ uint64_t smem_desc(uint32_t saddr) {
  uint64_t d = 0;
  d |= (uint64_t)((saddr & 0x3ffffu) >> 4);  // start address
  d |= (uint64_t)1 << 16;                    // leading byte offset (unused when swizzled)
  d |= (uint64_t)(1024 >> 4) << 32;          // stride byte offset
  d |= (uint64_t)1 << 46;                    // descriptor version
  d |= (uint64_t)2 << 61;                    // 128-byte swizzle
  return d;
}

// 16-byte asynchronous copy global -> shared (L2 only): copies src_bytes
// (0 or 16) from gsrc and fills the rest of the 16 bytes with zeros; with 0
// nothing is read.
__device__ __forceinline__ void cp_async16_zfill(uint32_t sdst, const void* gsrc, uint32_t src_bytes) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(sdst), "l"(gsrc), "r"(src_bytes)
               : "memory");
}
__device__ __forceinline__ void cp_async_wait_all() { asm volatile("cp.async.wait_all;" ::: "memory"); }
// One arrival on `bar` once every cp.async this thread issued so far has
// landed; the barrier's expected count includes it (.noinc).
__device__ __forceinline__ void cp_async_arrive_noinc(uint64_t* bar) {
  asm volatile("cp.async.mbarrier.arrive.noinc.shared::cta.b64 [%0];" ::"r"(smem_addr(bar)) : "memory");
}
__device__ __forceinline__ void tc_fence_before() {
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_addr(bar)) : "memory");
}

// 32 lanes x 32 consecutive fp32 columns of TMEM into registers.
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, uint32_t (&v)[32]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
      "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
      "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
      : "=r"(v[0]), "=r"(v[1]), "=r"(v[2]), "=r"(v[3]), "=r"(v[4]), "=r"(v[5]), "=r"(v[6]),
        "=r"(v[7]), "=r"(v[8]), "=r"(v[9]), "=r"(v[10]), "=r"(v[11]), "=r"(v[12]), "=r"(v[13]),
        "=r"(v[14]), "=r"(v[15]), "=r"(v[16]), "=r"(v[17]), "=r"(v[18]), "=r"(v[19]),
        "=r"(v[20]), "=r"(v[21]), "=r"(v[22]), "=r"(v[23]), "=r"(v[24]), "=r"(v[25]),
        "=r"(v[26]), "=r"(v[27]), "=r"(v[28]), "=r"(v[29]), "=r"(v[30]), "=r"(v[31])
      : "r"(taddr));
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}

// Drain one 128 x 256 fp32 accumulator to bf16 rows of Y.  Epilogue warp ew
// owns TMEM lanes 32ew .. 32ew+31 (rows r0 + 32ew ..); 64 columns at a time,
// each lane converts its row (nearest-even) into the warp's padded staging
// tile, then the warp stores it back out as 4 rows x 128 bytes per
// instruction.  Only rows below nvalid (owned by a route) are stored.
__device__ __forceinline__ void store_accumulator(uint32_t tcol, int ew, int lane, uint8_t* stage,
                                                  __nv_bfloat16* Y, int N, int r0, int n0, int nvalid) {
#pragma unroll 1
  for (int c2 = 0; c2 < BN / 64; ++c2) {
    uint4 out[8];
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      uint32_t v[32];
      tmem_ld32(tcol + (uint32_t)(64 * c2 + 32 * h), v);
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        float f[8];
#pragma unroll
        for (int i = 0; i < 8; ++i) f[i] = __uint_as_float(v[8 * q + i]);
        out[4 * h + q] = Vec<__nv_bfloat16>::from_float(f);
      }
    }
    uint4* srow = reinterpret_cast<uint4*>(stage + lane * kStageRowBytes);
#pragma unroll
    for (int q = 0; q < 8; ++q) srow[q] = out[q];
    __syncwarp();
    const int ch = lane & 7;
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const int row = 4 * i + (lane >> 3);
      const int col = n0 + 64 * c2 + 8 * ch;  // N % 8 == 0: a 16-byte chunk is wholly in or out
      if (32 * ew + row < nvalid && col < N) {
        const uint4 val = *reinterpret_cast<const uint4*>(stage + row * kStageRowBytes + ch * 16);
        *reinterpret_cast<uint4*>(Y + (size_t)(r0 + 32 * ew + row) * N + col) = val;
      }
    }
    __syncwarp();  // the staging tile is rewritten by the next 64 columns
  }
}

// Unit u -> expert x, first row r0 and owned rows of its 128-row block, and
// the column tile n0.  s_blk[x] = blocks of the experts before x.
struct Unit {
  int x, r0, nvalid, n0;
};

__device__ __forceinline__ Unit decode_unit(int u, int ntn, const int* s_blk, const int* s_off,
                                            const int* s_cnt, int e) {
  const int b = u / ntn;
  int lo = 0, hi = e;  // s_blk[lo] <= b < s_blk[hi]
  while (hi - lo > 1) {
    const int mid = (lo + hi) >> 1;
    if (s_blk[mid] <= b) lo = mid; else hi = mid;
  }
  Unit t;
  const int i = b - s_blk[lo];
  t.x = lo;
  t.r0 = s_off[lo] + BM * i;
  const int left = s_cnt[lo] - BM * i;
  t.nvalid = left < BM ? left : BM;
  t.n0 = (u - b * ntn) * BN;
  return t;
}

// ---- two-SM form (cta_group::2) ------------------------------------------
// A cluster of two CTAs on two SMs computes one 256 x 256 tile: CTA rank c
// holds rows 128c .. 128c+127 of the 256-row block (its A half) and columns
// 128c .. 128c+127 of the 256-column tile (its B half); one thread of rank
// 0 issues tcgen05.mma.cta_group::2 (M256 N256 K16), which reads both
// CTAs' shared memory at the same offsets and leaves each CTA's 128 rows
// of the fp32 result in its own TMEM.  Per SM and K-block only 32 KB move
// (48 KB in the one-SM form), so the ring holds six K-blocks.
//   both ranks, warp 0 lane 0: TMA of its A and B halves; the completion
//     bytes of both ranks are counted on rank 0's full barrier (the
//     .cta_group::2 form of the copy lets rank 1 signal it);
//   rank 0, warp 1 lane 0: MMA; its commits arrive on the empty / tfull
//     barriers of both ranks (multicast);
//   both ranks, warp 2: one collective TMEM allocation for the pair;
//   both ranks, warps 4..7: epilogue of its own rows, then an arrival on
//     rank 0's tempty barrier (remote for rank 1);
//   fused form, both ranks, warps 8..15: gather the CTA's 128 A rows, each
//     thread's copies arriving through cp.async.mbarrier.arrive.noinc;
//   fused form, rank 1, warp 1 lane 0: forwards each gathered stage to
//     rank 0's full barrier.
// A ring stage holds two 64-wide K blocks of this CTA's A and B halves (16 KB
// each per block), in a 3-stage ring: half the barrier round trips per MMA
// of one block per stage (measured 3-10 % faster for the plain form, 10-15 %
// for the fused one).
constexpr int kSubA = BM * BK * 2;              // 16 KB: 128 rows x 64 K of A, one swizzle atom column
constexpr int kSubB = (BN / 2) * BK * 2;        // 16 KB: 128 rows x 64 K of B
constexpr int kPairKB = 2;
constexpr int kPairStages = 3;
constexpr int kPairRingBytes = kPairStages * kPairKB * (kSubA + kSubB);  // 192 KB
constexpr int kPairSmemBytes = kPairRingBytes + kEpiBytes + 1024;
constexpr int BM2 = 2 * BM;                     // rows of a pair block

__device__ __forceinline__ uint32_t cluster_ctarank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}

// Address of the same shared-memory location in CTA `rank` of the cluster.
__device__ __forceinline__ uint32_t mapa_shared(uint32_t saddr, uint32_t rank) {
  uint32_t r;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(saddr), "r"(rank));
  return r;
}

__device__ __forceinline__ void cluster_sync_all() {
  asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::
                   : "memory");
}

// 2-D tile into this CTA's shared memory; completion bytes counted on the
// mbarrier at cluster address `mbar` (rank 0's barrier for both ranks).
__device__ __forceinline__ void tma_load_2d_pair(void* sdst, const CUtensorMap* map, int x, int y,
                                                 uint32_t mbar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.cta_group::2.shared::cluster.global.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%2, %3}], [%4];" ::"r"(smem_addr(sdst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(mbar)
      : "memory");
}

__device__ __forceinline__ void mma_bf16_pair(uint32_t dtmem, uint64_t adesc, uint64_t bdesc,
                                              uint32_t idesc, int accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::2.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(dtmem),
      "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
      : "memory");
}

// Arrive on the barrier at this offset in the CTAs of the pair that `mask`
// names (bit c = rank c) once the issuing thread's earlier MMAs have
// completed.
__device__ __forceinline__ void mma_commit_pair(uint64_t* bar, uint16_t mask = 0x3) {
  asm volatile(
      "tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64"
      " [%0], %1;" ::"r"(smem_addr(bar)),
      "h"(mask)
      : "memory");
}

// Bounded wait with cluster-scope acquire, for barriers that receive
// arrivals from the other CTA of the pair.
__device__ __forceinline__ bool mbar_wait_cluster(uint64_t* bar, uint32_t parity, uint64_t deadline_ns) {
  for (uint32_t it = 0;; ++it) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.acquire.cluster.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(smem_addr(bar)), "r"(parity)
        : "memory");
    if (ok) return true;
    if ((it & 63) == 63 && globaltimer_ns() > deadline_ns) return false;
  }
}

// 16 bytes from this CTA's shared memory to `dst` in another CTA of the
// cluster, the bytes counted on the mbarrier `mbar` there: a signal that
// travels through the async proxy (no cluster-scope release fence).
__device__ __forceinline__ void bulk_signal_s2s(uint32_t dst, const void* src, uint32_t mbar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.shared::cta.mbarrier::complete_tx::bytes [%0], [%1], 16, [%2];" ::"r"(dst),
      "r"(smem_addr(src)), "r"(mbar)
      : "memory");
}

__device__ __forceinline__ void mbar_arrive_cluster(uint32_t mbar) {
  asm volatile("mbarrier.arrive.release.cluster.shared::cluster.b64 _, [%0];" ::"r"(mbar) : "memory");
}

__device__ __forceinline__ uint32_t mma_idesc_pair() {
  uint32_t d = 0;
  d |= 1u << 4;                        // accumulator format: f32
  d |= 1u << 7;                        // A format: bf16
  d |= 1u << 10;                       // B format: bf16
  d |= (uint32_t)(BN >> 3) << 17;      // N / 8 (the pair's 256 columns)
  d |= (uint32_t)(BM2 >> 4) << 24;     // M / 16 (the pair's 256 rows)
  return d;
}

template <bool kGather>
__global__ void __launch_bounds__(kGather ? kGatherThreads : kThreads, 1)
    grouped_gemm_pair_kernel(const __grid_constant__ CUtensorMap tmA,
                             const __grid_constant__ CUtensorMap tmB, const GemmParams p) {
  constexpr int kPairABytes = kPairKB * kSubA;  // this CTA's 128 rows of A
  constexpr int kPairBBytes = kPairKB * kSubB;  // this CTA's 128 rows of B
  constexpr int kPairStageBytes = kPairABytes + kPairBBytes;
  extern __shared__ uint8_t smem_raw[];
  __shared__ __align__(8) uint64_t full[kPairStages], empty[kPairStages], tfull[2], tempty[2];
  __shared__ __align__(8) uint64_t gathered[kPairStages];  // fused form, rank 1: its gathered rows landed
  __shared__ __align__(8) uint64_t mma_drain;               // rank 0, after a time-out: its MMAs are done
  __shared__ __align__(16) uint8_t s_signal[16];             // fused form: source / target of rank 1's signal
  __shared__ uint32_t tmem_base;
  __shared__ int s_off[kMaxE + 1], s_cnt[kMaxE], s_blk[kMaxE + 1];
  __shared__ int s_err;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t rank = cluster_ctarank();  // 0 or 1 within the pair
  constexpr int kGatherWarps = (kGatherThreads - kThreads) / 32;
  constexpr int kGatherArrivals = kGatherWarps * 32;  // one per gathering thread and stage
  // identical static layout in both CTAs: the dynamic buffer starts at the
  // same offset, so the MMA's descriptors address the same tiles in both
  uint8_t* smem = smem_raw + ((1024 - (smem_addr(smem_raw) & 1023)) & 1023);
  const uint64_t deadline = globaltimer_ns() + (uint64_t)p.timeout_ns;

  for (int x = threadIdx.x; x <= p.e; x += blockDim.x) s_off[x] = __ldg(p.offsets + x);
  for (int x = threadIdx.x; x < p.e; x += blockDim.x) s_cnt[x] = __ldg(p.counts + x);
  if (threadIdx.x == 0) {
    s_err = 0;
    for (int i = 0; i < kPairStages; ++i) {
      // rank 0: its expect_tx arrival (both ranks' TMA bytes, and in the fused
      // form rank 1's 16-byte signal), plus its gathering threads' arrivals
      mbar_init(&full[i], kGather ? 1 + kGatherArrivals : 1);
      mbar_init(&empty[i], 1);  // the MMA commit, multicast to both ranks
      mbar_init(&gathered[i], kGatherArrivals);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&tfull[i], 1);
      mbar_init(&tempty[i], 2 * 4);  // rank 0: the epilogue warps of both ranks
    }
    mbar_init(&mma_drain, 1);
    fence_barrier_init();
  }
  __syncthreads();
  if (warp == 2) {
    asm volatile("tcgen05.alloc.cta_group::2.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                     smem_addr(&tmem_base)),
                 "r"(kTmemCols)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::2.sync.aligned;" ::: "memory");
  } else if (warp == 3) {
    // exclusive prefix over experts of their 256-row block counts
    int carry = 0;
    for (int x0 = 0; x0 < p.e; x0 += 32) {
      const int x = x0 + lane;
      const int c = x < p.e ? s_cnt[x] : 0;
      const int blocks = c > 0 ? (c + BM2 - 1) / BM2 : 0;
      int v = blocks;
#pragma unroll
      for (int d = 1; d < 32; d <<= 1) {
        const int w = __shfl_up_sync(0xffffffffu, v, d);
        if (lane >= d) v += w;
      }
      if (x < p.e) s_blk[x] = carry + v - blocks;
      carry += __shfl_sync(0xffffffffu, v, 31);
    }
    if (lane == 0) s_blk[p.e] = carry;
  }
  tc_fence_before();
  __syncthreads();
  cluster_sync_all();  // both ranks' barriers are initialised before any remote signal
  tc_fence_after();
  const uint32_t tbase = tmem_base;

  const int ntn = (p.N + BN - 1) / BN;  // the last column tile may be partial
  const int nunits = s_blk[p.e] * ntn;
  const int kblocks = (p.K + BK * kPairKB - 1) / (BK * kPairKB);  // per stage; columns past K read as zeros
  const int pair = blockIdx.x >> 1, npairs = gridDim.x >> 1;

  if (warp == 0 && lane == 0) {
    // ---- TMA producer (both ranks) ---------------------------------------
    int stage = 0;
    uint32_t phase = 0;
    bool ok = true;
    for (int u = pair; u < nunits && ok; u += npairs) {
      const Unit t = decode_unit(u, ntn, s_blk, s_off, s_cnt, p.e);  // rows in units of BM2 below
      const int b = u / ntn;
      const int r0 = s_off[t.x] + BM2 * (b - s_blk[t.x]) + BM * (int)rank;
      for (int kb = 0; kb < kblocks; ++kb) {
        if (!mbar_wait_bounded(&empty[stage], phase ^ 1u, deadline)) {
          ok = false;
          break;
        }
        uint8_t* sa = smem + stage * kPairStageBytes;
        const uint32_t fb = mapa_shared(smem_addr(&full[stage]), 0);
        if (rank == 0) mbar_arrive_expect_tx(&full[stage], kGather ? 2 * kPairBBytes + 16 : 2 * kPairStageBytes);
#pragma unroll
        for (int q = 0; q < kPairKB; ++q) {
          const int kx = (kb * kPairKB + q) * BK;
          if (!kGather) tma_load_2d_pair(sa + q * kSubA, &tmA, kx, r0, fb);
          tma_load_2d_pair(sa + kPairABytes + q * kSubB, &tmB, kx, t.x * p.N + t.n0 + (BN / 2) * (int)rank, fb);
        }
        if (++stage == kPairStages) {
          stage = 0;
          phase ^= 1u;
        }
      }
    }
    // drain: every stage's last fill consumed, so no commit of rank 0 is
    // still on its way to this CTA's barriers when it leaves
    for (int i = 0; i < kPairStages && ok; ++i) {
      if (!mbar_wait_bounded(&empty[stage], phase ^ 1u, deadline)) ok = false;
      if (++stage == kPairStages) {
        stage = 0;
        phase ^= 1u;
      }
    }
    if (!ok) atomicOr(&s_err, 1);
  } else if (kGather && warp >= kThreads / 32) {
    // ---- A gather (fused form, both ranks): this CTA's 128 rows ------------
    // Each lane copies 16 bytes of kGatherRows / 4 rows per K block (8 lanes per 128-byte
    // row, the swizzle as in the one-SM form), then hands its copies of the
    // stage to the stage's barrier (cp.async.mbarrier.arrive.noinc: one
    // arrival once they land) and runs on to the next free stage; waiting
    // for its own copies two stages later instead held the gather to a
    // shallow window and the fused GEMM 10-15 % lower.  Rank 0's threads
    // arrive on its full barrier, rank 1's on its own `gathered` barrier,
    // forwarded below; the waiter on each fences the async proxy.  A unit's
    // row-to-token indices are loaded while the previous unit is gathered.
    const int gw = warp - kThreads / 32, chunk = lane & 7;
    int stage = 0;
    uint32_t phase = 0;
    bool ok = true;
    // token of each of this lane's kGatherRows / 4 rows in unit u; -1 for rows no route owns
    auto unit_tokens = [&](int u, int* tok) {
      const Unit t = decode_unit(u, ntn, s_blk, s_off, s_cnt, p.e);
      const int i = u / ntn - s_blk[t.x];
      const int r0 = s_off[t.x] + BM2 * i + BM * (int)rank;
      const int left = s_cnt[t.x] - BM2 * i - BM * (int)rank;
#pragma unroll
      for (int j = 0; j < kGatherRows / 4; ++j) {
        const int rr = kGatherRows * gw + 4 * j + (lane >> 3);
        tok[j] = -1;
        if (rr < left) {
          const int v = __ldg(p.inv_row + r0 + rr);
          tok[j] = (unsigned)v < (unsigned)p.s ? v : 0;
        }
      }
    };
    int tok[kGatherRows / 4], ntok[kGatherRows / 4];
#pragma unroll
    for (int j = 0; j < kGatherRows / 4; ++j) ntok[j] = -1;  // after the last unit: nothing
    if (pair < nunits) unit_tokens(pair, tok);
    for (int u = pair; u < nunits && ok; u += npairs) {
      if (u + npairs < nunits) unit_tokens(u + npairs, ntok);  // in flight while this unit is gathered
      const __nv_bfloat16* src[kGatherRows / 4];
#pragma unroll
      for (int j = 0; j < kGatherRows / 4; ++j) src[j] = p.x + (size_t)(tok[j] < 0 ? 0 : tok[j]) * p.K + chunk * 8;
      for (int kb = 0; kb < kblocks; ++kb) {
        bool waited = true;
        if (lane == 0) waited = mbar_wait_bounded(&empty[stage], phase ^ 1u, deadline);
        if (!__shfl_sync(0xffffffffu, waited ? 1 : 0, 0)) {
          ok = false;
          break;
        }
        const uint32_t sa = smem_addr(smem + stage * kPairStageBytes);
#pragma unroll
        for (int q = 0; q < kPairKB; ++q) {
          const int kx = (kb * kPairKB + q) * BK;
#pragma unroll
          for (int j = 0; j < kGatherRows / 4; ++j) {
            // rows no route owns are not copied (their results are never stored)
            const int rr = kGatherRows * gw + 4 * j + (lane >> 3);
            if (tok[j] >= 0) {
              // columns past K: zeros, nothing read (the row's end may be the buffer's)
              const bool in_k = kx + chunk * 8 < p.K;
              cp_async16_zfill(sa + q * kSubA + rr * 128 + ((chunk ^ (rr & 7)) << 4), in_k ? src[j] + kx : src[j],
                               in_k ? 16u : 0u);
            }
          }
        }
        cp_async_arrive_noinc(rank == 0 ? &full[stage] : &gathered[stage]);
        if (++stage == kPairStages) {
          stage = 0;
          phase ^= 1u;
        }
      }
#pragma unroll
      for (int j = 0; j < kGatherRows / 4; ++j) tok[j] = ntok[j];
    }
    cp_async_wait_all();  // nothing of this thread's stays in flight
    if (!ok && lane == 0) atomicOr(&s_err, 1);
  } else if (kGather && warp == 1 && lane == 0 && rank == 1) {
    // ---- forwarder (fused form, rank 1) ------------------------------------
    // Once all of this CTA's gathering warps have landed a stage, a 16-byte
    // shared-to-shared bulk copy into rank 0 counts on rank 0's full barrier:
    // an async-proxy signal, ordered after the gathered rows (fenced by
    // their writers, acquired here through the `gathered` barrier).
    const uint32_t sig_dst = mapa_shared(smem_addr(s_signal), 0);
    int stage = 0;
    uint32_t phase = 0;
    bool ok = true;
    for (int u = pair; u < nunits && ok; u += npairs) {
      for (int kb = 0; kb < kblocks; ++kb) {
        if (!mbar_wait_bounded(&gathered[stage], phase, deadline)) {
          ok = false;
          break;
        }
        fence_proxy_async_smem();  // the rows landed by cp.async, before the async-proxy signal
        bulk_signal_s2s(sig_dst, s_signal, mapa_shared(smem_addr(&full[stage]), 0));
        if (++stage == kPairStages) {
          stage = 0;
          phase ^= 1u;
        }
      }
    }
    if (!ok) atomicOr(&s_err, 1);
  } else if (warp == 1 && lane == 0 && rank == 0) {
    // ---- MMA issuer (rank 0) ----------------------------------------------
    const uint32_t idesc = mma_idesc_pair();
    int stage = 0, acc = 0;
    uint32_t phase = 0, tphase[2] = {0u, 0u};
    bool ok = true;
    for (int u = pair; u < nunits && ok; u += npairs) {
      if (!mbar_wait_cluster(&tempty[acc], tphase[acc] ^ 1u, deadline)) {
        ok = false;
        break;
      }
      tphase[acc] ^= 1u;
      tc_fence_after();
      const uint32_t dt = tbase + (uint32_t)(acc * BN);
      for (int kb = 0; kb < kblocks; ++kb) {
        if (!mbar_wait_cluster(&full[stage], phase, deadline)) {
          ok = false;
          break;
        }
        tc_fence_after();
        if (kGather) fence_proxy_async_smem();  // this CTA's rows landed by cp.async
        const uint32_t sa = smem_addr(smem + stage * kPairStageBytes);
#pragma unroll
        for (int q = 0; q < kPairKB; ++q) {
          const uint64_t ad = smem_desc(sa + q * kSubA), bd = smem_desc(sa + kPairABytes + q * kSubB);
#pragma unroll
          for (int kk = 0; kk < BK / 16; ++kk)
            mma_bf16_pair(dt, ad + (uint64_t)(2 * kk), bd + (uint64_t)(2 * kk), idesc, (kb | q | kk) != 0);
        }
        mma_commit_pair(&empty[stage]);
        if (++stage == kPairStages) {
          stage = 0;
          phase ^= 1u;
        }
      }
      if (!ok) break;
      mma_commit_pair(&tfull[acc]);
      acc ^= 1;
    }
    if (!ok) {
      // a wait ran out: before this CTA (and, at the cluster barrier below,
      // its partner) leaves, let every MMA issued so far finish reading both
      // CTAs' shared memory -- one more commit, to this CTA only, arrives
      // after all of them and after the commits before it (bounded wait)
      mma_commit_pair(&mma_drain, 0x1);
      mbar_wait_bounded(&mma_drain, 0, globaltimer_ns() + (uint64_t)p.timeout_ns);
      atomicOr(&s_err, 1);
    }
  } else if (warp >= 4 && warp < 8) {
    // ---- epilogue (both ranks): own 128 rows ------------------------------
    const int ew = warp - 4;
    const uint32_t te0 = mapa_shared(smem_addr(&tempty[0]), 0), te1 = mapa_shared(smem_addr(&tempty[1]), 0);
    int acc = 0;
    uint32_t tphase[2] = {0u, 0u};
    bool ok = true;
    for (int u = pair; u < nunits && ok; u += npairs) {
      const Unit t = decode_unit(u, ntn, s_blk, s_off, s_cnt, p.e);
      const int b = u / ntn;
      const int i = b - s_blk[t.x];
      const int r0 = s_off[t.x] + BM2 * i + BM * (int)rank;
      const int left = s_cnt[t.x] - BM2 * i - BM * (int)rank;
      const int nvalid = left < 0 ? 0 : (left < BM ? left : BM);
      // every lane waits (and acquires) itself; the warp leaves together
      if (!__all_sync(0xffffffffu, mbar_wait_bounded(&tfull[acc], tphase[acc], deadline))) {
        ok = false;
        break;
      }
      tphase[acc] ^= 1u;
      tc_fence_after();
      store_accumulator(tbase + ((uint32_t)(32 * ew) << 16) + (uint32_t)(acc * BN), ew, lane,
                        smem + kPairStages * kPairStageBytes + ew * kEpiWarpBytes, p.Y, p.N, r0, t.n0, nvalid);
      tc_fence_before();
      __syncwarp();  // every lane's TMEM reads are done
      if (lane == 0) {
        if (rank == 0) mbar_arrive(&tempty[acc]);
        else mbar_arrive_cluster(acc ? te1 : te0);
      }
      acc ^= 1;
    }
    if (!ok) atomicOr(&s_err, 1);
  }

  tc_fence_before();
  __syncthreads();
  cluster_sync_all();  // both ranks done with TMEM and with each other's barriers
  tc_fence_after();
  if (warp == 2)
    asm volatile("tcgen05.dealloc.cta_group::2.sync.aligned.b32 %0, %1;" ::"r"(tbase),
                 "r"(kTmemCols)
                 : "memory");
  if (threadIdx.x == 0 && s_err) raise_status(p.status, MOE_DEV_TIMEOUT);
}

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  // a function-local static initialises once, thread-safe
  static const PFN_cuTensorMapEncodeTiled_v12000 fn = [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      return reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
    return static_cast<PFN_cuTensorMapEncodeTiled_v12000>(nullptr);
  }();
  return fn;
}

// 2-D bf16 row-major [outer, inner] tensor, box (BK inner) x box_rows, 128-B swizzle.
bool make_map(CUtensorMap* map, const void* base, uint64_t inner, uint64_t outer, uint32_t box_rows) {
  auto fn = encode_fn();
  if (!fn) return false;
  cuuint64_t dims[2] = {inner, outer};
  cuuint64_t strides[1] = {inner * 2};
  cuuint32_t box[2] = {BK, box_rows};
  cuuint32_t estride[2] = {1, 1};
  return fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box,
            estride, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

template <bool kGather>
cudaError_t launch_pair(const CUtensorMap& ma, const CUtensorMap& mb, const GemmParams& p,
                        const DeviceInfo& di, cudaStream_t st) {
  static OncePerDevice once;
  cudaError_t err = once.run([] {
    return cudaFuncSetAttribute(grouped_gemm_pair_kernel<kGather>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                kPairSmemBytes);
  });
  if (err != cudaSuccess) return err;
  // pair units: at most ceil(rows / 256) + e blocks of 256 rows, times the column tiles
  const long long units = (((long long)p.rows + BM2 - 1) / BM2 + p.e) * ((p.N + BN - 1) / BN);
  long long pairs = di.sms / 2;
  if (units < pairs) pairs = units;
  if (pairs < 1) pairs = 1;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)(2 * pairs));
  cfg.blockDim = dim3(kGather ? kGatherThreads : kThreads);
  cfg.dynamicSmemBytes = kPairSmemBytes;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 2;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, grouped_gemm_pair_kernel<kGather>, ma, mb, p);
}

GemmParams params(const int32_t* offsets, const int32_t* counts, int e, int rows, int K, int N,
                  void* Y, int32_t* status) {
  GemmParams p;
  p.x = nullptr;
  p.offsets = offsets;
  p.counts = counts;
  p.inv_row = nullptr;
  p.e = e;
  p.rows = rows;
  p.K = K;
  p.N = N;
  p.s = 0;
  p.Y = static_cast<__nv_bfloat16*>(Y);
  p.status = status;
  p.timeout_ns = 2000000000LL;
  return p;
}

}  // namespace

cudaError_t launch_grouped_gemm(const int32_t* offsets, const int32_t* counts, int e, int rows, int K,
                                int N, const void* X, const void* W, void* Y, int32_t* status,
                                const DeviceInfo& di, cudaStream_t st) {
  CUtensorMap ma, mb;
  if (!make_map(&ma, X, (uint64_t)K, (uint64_t)rows, BM) ||
      !make_map(&mb, W, (uint64_t)K, (uint64_t)e * (uint64_t)N, BN / 2))
    return cudaErrorInvalidValue;
  return launch_pair<false>(ma, mb, params(offsets, counts, e, rows, K, N, Y, status), di, st);
}

cudaError_t launch_dispatch_gemm(const int32_t* offsets, const int32_t* counts, const int32_t* inv_row,
                                 int e, int rows, int s, int K, int N, const void* x, const void* W,
                                 void* Y, int32_t* status, const DeviceInfo& di, cudaStream_t st) {
  CUtensorMap mb;
  GemmParams p = params(offsets, counts, e, rows, K, N, Y, status);
  p.x = static_cast<const __nv_bfloat16*>(x);
  p.inv_row = inv_row;
  p.s = s;
  if (!make_map(&mb, W, (uint64_t)K, (uint64_t)e * (uint64_t)N, BN / 2)) return cudaErrorInvalidValue;
  return launch_pair<true>(mb, mb, p, di, st);  // A is gathered by threads: no A map
}

}  // namespace moe
