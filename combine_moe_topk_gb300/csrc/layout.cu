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
//   B. decoupled look-back over tiles: each tile publishes its aggregate
//      (per expert a 32-bit word: the count, and the published flag in its
//      top bit) as soon as its histogram is done,
//      then reads the aggregates of all its predecessors at once -- groups of
//      threads per expert, eight independent loads in flight each -- instead
//      of walking back one tile at a time, so the look-back costs a few L2
//      round trips whatever the tile count.  The same pass over all tiles
//      gives the global expert totals, which dropless rows need everywhere
//      and the last tile writes out;
//   C. slots: per sub-tile, each warp builds a 32-bit token mask per expert
//      (atomicOr: order-free), so a route's rank among the warp's tokens is
//      popc(mask & lanes-below); warps are scanned in order per expert.
// All waits are bounded on the global timer; when one runs out the kernel
// records MOE_DEV_TIMEOUT and carries on with what it has (no hang, no trap).
// All tiles are co-resident (cooperative launch), which is what makes the
// wait for the last tile safe.
//
// Rebuilds.  A handle's layout can be rebuilt in place from new routes with
// no allocation and no memset: a look-back word counts as published when its
// top bit equals the build's parity, and every build rewrites every tile's
// row, so the previous build's rows read as unpublished.  The parity is
// found on the device, not passed in (so a CUDA graph that replays a build
// stays right): each tile reads the top bit of its own row, which only it
// writes -- zero after the allocation's memset, else the previous build's
// parity -- and takes the other value.  Tile 0 clears the status word and
// the rank counts before it publishes; every other tile reads tile 0's row
// before its own atomics.
//
// Fused gate (e <= 32).  With router logits instead of expert ids, phase A
// first selects each token's experts in the token's own thread (all the
// tile's logits loaded at once; topk_token_thread gives the gate kernel's
// ids and gate bits) and writes the ids and gates out.  It is instantiated
// for e <= 8 and e <= 32, so a small router's thread runs through 8-wide
// loops (the fused kernel took 9.6 us alone on 256 tokens over 8 experts
// with 32-wide ones, 8.0 us with 8-wide).  For more experts a
// thread per token holds too many logits, and a warp per token inside a
// tile selects its 32 tokens one after another: measured slower than the
// gate kernel followed by the layout kernel, which is what runs there.
#include <atomic>
#include <initializer_list>
#include <mutex>

#include "common.cuh"
#include "gate_core.cuh"
#include "internal.h"

namespace moe {

namespace {

constexpr int kThreads = 256;  // also the sub-tile size in tokens
constexpr int kWarps = kThreads / 32;
constexpr int kMaxE = 256;
constexpr int kMaxK = 16;
constexpr int kMaxR = 64;

// Look-back word: the published flag in bit 31, the tile's route count for
// one expert in bits 0-30 (a count never exceeds s < 2^31).  Rows of e
// words are padded to a multiple of four so they can be read as 16-byte
// vectors.
constexpr unsigned kPublished = 0x80000000u;
constexpr int kLookbackLoads = 8;        // 16-byte look-back loads in flight per thread
constexpr int kMaxLookbackWords = 16384;  // tiles * padded e, at most: bounds the look-back reads

__host__ __device__ inline int padded_e(int e) { return (e + 3) & ~3; }

// The scan runs over "units" in priority order.  Token-major priority: a
// unit is a token with its k routes.  k-major priority (every first choice
// before any second choice): a unit is one route, units ordered slot by slot,
// so the same token-order scan over s*k one-route units gives k-major slots.
struct Params {
  const int32_t* topk_idx;
  int s, e, k;           // units, experts, routes per unit
  int s_tok, k_tok;      // tokens and routes per token of the caller's arrays
  int kmajor;            // units are single routes in slot-major order
  int capacity, R;       // R: dedup ranks counted in this kernel (0 in k-major mode)
  int R_tok;             // the caller's dedup rank count
  int pad;               // dropless rows per expert padded to a multiple of pad
  int tiles, subtiles_per_tile;
  LayoutOut out;
  int hold_tile;
  long long timeout_ns;
  int clear_status;      // tile 0 clears the status word and the rank counts
  int absent_ok;         // an expert id of -1 is a route that does not exist (not an error)
  int rows;              // rows of the dispatched buffer: no route gets a row at or past it
  // fused gate (layout_kernel with EPL > 0): router logits [s, e] in, the
  // caller's ids [s, k] and gates [s, k] out
  const float* logits;
  int renorm;
  int32_t* gate_idx;
  float* gate_val;
};

// Index of unit v's first route in the caller's [s_tok, k_tok] arrays.
__device__ __forceinline__ size_t unit_base(const Params& p, int v) {
  if (!p.kmajor) return (size_t)v * p.k;
  const int j = v / p.s_tok;
  return (size_t)(v - j * p.s_tok) * p.k_tok + j;
}

__device__ __forceinline__ uint4 ld_relaxed_v4(const uint4* p) {
  uint4 v;
  asm volatile("ld.relaxed.gpu.global.v4.u32 {%0,%1,%2,%3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "l"(p)
               : "memory");
  return v;
}

__device__ __forceinline__ unsigned ld_relaxed_u32(const unsigned* p) {
  unsigned v;
  asm volatile("ld.relaxed.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}

__device__ __forceinline__ unsigned ld_acquire_u32(const unsigned* p) {
  unsigned v;
  asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}

__device__ __forceinline__ void st_relaxed_u32(unsigned* p, unsigned v) {
  asm volatile("st.relaxed.gpu.global.u32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}

// All four words carry this build's publish bit (pub = kPublished or 0).
__device__ __forceinline__ bool all_published(const uint4& w, unsigned pub) {
  const unsigned x = pub ? (w.x & w.y & w.z & w.w) : ~(w.x | w.y | w.z | w.w);
  return (x & kPublished) != 0;
}

// Load token t's k expert ids (16- or 8-byte loads when k allows) and mark
// which routes are valid: in range and not a repeat of an earlier route of
// the same token.
template <int KM>
__device__ __forceinline__ unsigned load_routes(const Params& p, int t, int* xs, unsigned* absent) {
  const int32_t* src = p.topk_idx + unit_base(p, t);
  if ((p.k & 3) == 0) {
#pragma unroll
    for (int j4 = 0; j4 < (KM / 4); ++j4)
      if (4 * j4 < p.k) {
        const int4 v = __ldg(reinterpret_cast<const int4*>(src) + j4);
        xs[4 * j4] = v.x;
        xs[4 * j4 + 1] = v.y;
        xs[4 * j4 + 2] = v.z;
        xs[4 * j4 + 3] = v.w;
      }
  } else if ((p.k & 1) == 0) {
#pragma unroll
    for (int j2 = 0; j2 < (KM / 2); ++j2)
      if (2 * j2 < p.k) {
        const int2 v = __ldg(reinterpret_cast<const int2*>(src) + j2);
        xs[2 * j2] = v.x;
        xs[2 * j2 + 1] = v.y;
      }
  } else {
#pragma unroll
    for (int j = 0; j < KM; ++j)
      if (j < p.k) xs[j] = __ldg(src + j);
  }
  unsigned valid = 0, none = 0;
#pragma unroll
  for (int j = 0; j < KM; ++j) {
    if (j < p.k) {
      const int x = xs[j];
      bool ok = x >= 0 && x < p.e;
#pragma unroll
      for (int jj = 0; jj < j; ++jj)
        if (xs[jj] == x) ok = false;
      if (ok) valid |= 1u << j;
      if (p.absent_ok && x == -1) none |= 1u << j;
    }
  }
  *absent = none;
  return valid;
}

// Set bit `lane` of the warp's token mask of every valid route's expert.
template <int KM>
__device__ __forceinline__ void mark_routes(const Params& p, unsigned (*mask)[kMaxE], int warp,
                                            int lane, const int* xs, unsigned valid) {
#pragma unroll
  for (int j = 0; j < KM; ++j)
    if ((valid >> j) & 1u) atomicOr(&mask[warp][xs[j]], 1u << lane);
}

// Decoupled look-back with a full-width window.  Publishes this tile's
// aggregate row, then reads the rows of tiles [0, nread) -- each thread a
// column of four experts over a strided set of tiles, eight 16-byte loads in
// flight -- and adds them up: s_excl[x] gets the routes of tiles before this
// one, s_tot[x] (which holds this tile's own aggregate on entry) the routes
// of every tile read.  Waits are bounded; a time-out sets *timed_out and the
// missing rows count as empty.
__device__ void lookback(const Params& p, int tile, int nread, const int* s_agg, int* s_excl,
                         int* s_tot, unsigned pub, uint64_t deadline, bool* timed_out) {
  const int tid = threadIdx.x, lane = tid & 31;
  const int e4 = padded_e(p.e);
  unsigned* rows = reinterpret_cast<unsigned*>(p.out.lookback);
  // release: each of tile 0's threads fences its own clears (rank_counts[tid],
  // the status word for tid 0) before storing word tid of the row, which the
  // other tiles acquire before their atomics on the same index (no other
  // tile publishes anything another tile reads, and a lone tile's clears and
  // atomics are the same thread's, same address)
  if (tile == 0 && p.clear_status && p.tiles > 1) __threadfence();
  if (tile != p.hold_tile)
    for (int x = tid; x < e4; x += kThreads)
      st_relaxed_u32(rows + (size_t)tile * e4 + x, pub | (unsigned)(x < p.e ? s_agg[x] : 0));

  // a held tile (test hook) publishes one more time-out after its own
  // deadline -- well after every waiting tile has given up, whatever the
  // skew of the tiles' start times -- so that every build still rewrites
  // every row
  if (tile == p.hold_tile) {
    const uint64_t release_at = deadline + (uint64_t)p.timeout_ns;
    while (globaltimer_ns() <= release_at) __nanosleep(1000);
    for (int x = tid; x < e4; x += kThreads)
      st_relaxed_u32(rows + (size_t)tile * e4 + x, pub | (unsigned)(x < p.e ? s_agg[x] : 0));
  }
  // nothing to read: this tile's totals are its own, no earlier routes
  if (nread <= (tile < nread ? 1 : 0)) return;
  const int quads = e4 / 4;
  const int groups = kThreads / quads;  // threads (g, q) read tiles g, g + groups, ...
  const int g = tid / quads, q = tid - (tid / quads) * quads;
  unsigned ex[4] = {0, 0, 0, 0}, tot[4] = {0, 0, 0, 0};
  if (g < groups) {
    const uint4* col = reinterpret_cast<const uint4*>(rows) + q;  // row b at col[b * quads]
    for (int b0 = g; b0 < nread; b0 += groups * kLookbackLoads) {
      uint4 w[kLookbackLoads];
#pragma unroll
      for (int u = 0; u < kLookbackLoads; ++u) {
        const int b = b0 + groups * u;
        w[u] = (b < nread && b != tile) ? ld_relaxed_v4(col + (size_t)b * quads)
                                         : make_uint4(pub, pub, pub, pub);
      }
#pragma unroll
      for (int u = 0; u < kLookbackLoads; ++u) {
        const int b = b0 + groups * u;
        if (b >= nread || b == tile) continue;
        for (uint32_t it = 0; !all_published(w[u], pub) && !*timed_out; ++it) {
          __nanosleep(32);
          if ((it & 15) == 15 && globaltimer_ns() > deadline) *timed_out = true;
          w[u] = ld_relaxed_v4(col + (size_t)b * quads);
        }
        if (*timed_out && !all_published(w[u], pub)) continue;
        const unsigned v[4] = {w[u].x & ~kPublished, w[u].y & ~kPublished, w[u].z & ~kPublished,
                               w[u].w & ~kPublished};
#pragma unroll
        for (int c = 0; c < 4; ++c) {
          tot[c] += v[c];
          if (b < tile) ex[c] += v[c];
        }
      }
    }
  }
  // sum the lanes of the warp that read the same column (xor shuffles, when
  // the column count is a power of two), then shared atomics per column
  bool leader = g < groups;
  if (quads < 32 && (quads & (quads - 1)) == 0) {
    for (int off = quads; off < 32; off <<= 1)
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        ex[c] += __shfl_xor_sync(0xffffffffu, ex[c], off);
        tot[c] += __shfl_xor_sync(0xffffffffu, tot[c], off);
      }
    leader = lane < quads;
  }
  if (leader) {
#pragma unroll
    for (int c = 0; c < 4; ++c) {
      const int x = 4 * q + c;
      if (x < p.e) {
        atomicAdd(&s_excl[x], (int)ex[c]);
        atomicAdd(&s_tot[x], (int)tot[c]);
      }
    }
  }
}

// Per-expert exclusive scan of the counts (e <= 256: up to eight per lane of
// warp 0, then a warp scan) into s_off[0..e]; the tile that holds the totals of
// record also writes raw_counts, counts and offsets to the handle.
__device__ void expert_offsets(const Params& p, const int* s_tot, int* s_off, bool write_out) {
  const int lane = threadIdx.x & 31;
  if ((threadIdx.x >> 5) != 0) return;
  // lane l takes experts l*ipl .. l*ipl+ipl-1 (ipl = 1 for e <= 32, so a
  // small router's scan is one item per lane, not eight on lane 0)
  const int ipl = (p.e + 31) >> 5;
  int raw[8], v[8];
  int sum = 0;
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    const int x = lane * ipl + i;
    raw[i] = (i < ipl && x < p.e) ? s_tot[x] : 0;
    v[i] = p.capacity > 0 ? min(raw[i], p.capacity) : raw[i];
    sum += p.pad > 1 ? (v[i] + p.pad - 1) / p.pad * p.pad : v[i];  // rows of the expert's segment
  }
  int incl = sum;
#pragma unroll
  for (int off = 1; off < 32; off <<= 1) {
    const int o = __shfl_up_sync(0xffffffffu, incl, off);
    if (lane >= off) incl += o;
  }
  int run = incl - sum;
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    const int x = lane * ipl + i;
    if (i < ipl && x < p.e) {
      const int off = p.capacity > 0 ? x * p.capacity : run;
      s_off[x] = off;
      if (write_out) {
        // a segment is cut at the buffer's rows (a dropless bound below the
        // routes: the routes past it get no row, write_routes reports them)
        const int o = min(off, p.rows);
        p.out.raw_counts[x] = raw[i];
        p.out.counts[x] = min(v[i], p.rows - o);
        p.out.offsets[x] = o;
      }
    }
    run += p.pad > 1 ? (v[i] + p.pad - 1) / p.pad * p.pad : v[i];
  }
  if (lane == 31) {
    const int end = p.capacity > 0 ? p.e * p.capacity : run;
    s_off[p.e] = end;
    if (write_out) p.out.offsets[p.e] = min(end, p.rows);
  }
}

// Store k int32 values of one token (16- or 8-byte stores when k allows).
template <int KM>
__device__ __forceinline__ void store_route_ints(int32_t* dst, const int* v, int k) {
  if ((k & 3) == 0) {
#pragma unroll
    for (int j4 = 0; j4 < (KM / 4); ++j4)
      if (4 * j4 < k)
        reinterpret_cast<int4*>(dst)[j4] = make_int4(v[4 * j4], v[4 * j4 + 1], v[4 * j4 + 2], v[4 * j4 + 3]);
  } else if ((k & 1) == 0) {
#pragma unroll
    for (int j2 = 0; j2 < (KM / 2); ++j2)
      if (2 * j2 < k) reinterpret_cast<int2*>(dst)[j2] = make_int2(v[2 * j2], v[2 * j2 + 1]);
  } else {
#pragma unroll
    for (int j = 0; j < KM; ++j)
      if (j < k) dst[j] = v[j];
  }
}

// Write one token's routes: token-order slot, row, drop flag, and its
// virtual-rank set; with inv_row, the token number at each kept row.
// base[x] (+ excl[x] when given: the routes of earlier tiles) is the slot of
// this warp's first token routed to x; mask[x] the warp's token mask for x.
// Returns the token's rank set.
template <int KM>
__device__ __forceinline__ unsigned long long write_routes(const Params& p, int t, int lane,
                                                           const int* xs, unsigned valid,
                                                           const int* base, const int* excl,
                                                           const unsigned* mask, const int* s_off, bool* over) {
  const unsigned below = (1u << lane) - 1u;
  // experts per virtual rank, as a shift when a power of two
  const int per_rank = p.R > 0 ? p.e / p.R : 1;
  const int rank_shift = (per_rank & (per_rank - 1)) == 0 ? __ffs(per_rank) - 1 : -1;
  unsigned long long ranks = 0;
  int loc[KM], row[KM];
  uint32_t dropw[(KM + 3) / 4];
#pragma unroll
  for (int q = 0; q < (KM + 3) / 4; ++q) dropw[q] = 0;
#pragma unroll
  for (int j = 0; j < KM; ++j) {
    loc[j] = -1;
    row[j] = -1;
    if (j < p.k && ((valid >> j) & 1u)) {
      const int x = xs[j];
      const int l = base[x] + (excl ? excl[x] : 0) + __popc(mask[x] & below);
      loc[j] = l;
      if (p.capacity > 0) {
        if (l < p.capacity) row[j] = x * p.capacity + l;
      } else {
        row[j] = s_off[x] + l;
        if (row[j] >= p.rows) {  // past the caller's bound on the rows: not kept, reported
          row[j] = -1;
          *over = true;
        }
      }
      if (p.R > 0 && row[j] >= 0) ranks |= 1ull << (rank_shift >= 0 ? x >> rank_shift : x / per_rank);
    }
    if (row[j] < 0) dropw[j / 4] |= 1u << (8 * (j % 4));
  }
  const size_t q0 = unit_base(p, t);
  if (p.out.inv_row) {
    const int token = p.kmajor ? t - (t / p.s_tok) * p.s_tok : t;
#pragma unroll
    for (int j = 0; j < KM; ++j)
      if (j < p.k && row[j] >= 0) p.out.inv_row[row[j]] = token;
  }
  store_route_ints<KM>(p.out.loc + q0, loc, p.k);
  store_route_ints<KM>(p.out.row + q0, row, p.k);
  uint8_t* dr = p.out.drop + q0;
  if ((p.k & 3) == 0) {
#pragma unroll
    for (int j4 = 0; j4 < (KM / 4); ++j4)
      if (4 * j4 < p.k) reinterpret_cast<uint32_t*>(dr)[j4] = dropw[j4];
  } else {
#pragma unroll
    for (int j = 0; j < KM; ++j)
      if (j < p.k) dr[j] = (uint8_t)((dropw[j / 4] >> (8 * (j % 4))) & 0xffu);
  }
  if (p.R > 0) {
    uint8_t* tir = p.out.token_in_rank + (size_t)t * p.R;
    if ((p.R & 3) == 0) {  // four ranks' bytes per 4-byte store (t * R is a multiple of 4)
      for (int r = 0; r < p.R; r += 4) {
        const uint32_t b = (uint32_t)(ranks >> r) & 0xfu;
        *reinterpret_cast<uint32_t*>(tir + r) = (b & 1u) | ((b & 2u) << 7) | ((b & 4u) << 14) | ((b & 8u) << 21);
      }
    } else {
      for (int r = 0; r < p.R; ++r) tir[r] = (uint8_t)((ranks >> r) & 1ull);
    }
  }
  return ranks;
}

// Add the warp's rank sets into the per-rank token counts: one ballot per
// rank that any lane of the warp sends to.
__device__ __forceinline__ void count_ranks(unsigned long long ranks, int lane, int* s_rank) {
  const unsigned lo = __reduce_or_sync(0xffffffffu, (unsigned)ranks);
  const unsigned hi = __reduce_or_sync(0xffffffffu, (unsigned)(ranks >> 32));
  unsigned long long any = ((unsigned long long)hi << 32) | lo;
  while (any) {
    const int r = __ffsll((long long)any) - 1;
    any &= any - 1;
    const int n = __popc(__ballot_sync(0xffffffffu, (ranks >> r) & 1ull));
    if (lane == 0) atomicAdd(&s_rank[r], n);
  }
}

// Fused gate: thread t's token selects its experts (topk_token_thread, the
// gate kernel's ids and gate bits for e <= 32) and writes the ids and gates
// to the caller's arrays.  Returns whether a logit was not finite.
template <int KM, int EM>
__device__ __forceinline__ bool gate_thread_token(const Params& p, int t, int* xs) {
  float g[KM];
  const bool bad = topk_token_thread<KM, EM>(p.logits + (size_t)t * p.e, p.e, p.k, p.renorm, xs, g);
  store_route_ints<KM>(p.gate_idx + (size_t)t * p.k, xs, p.k);
  float* gd = p.gate_val + (size_t)t * p.k;
#pragma unroll
  for (int j = 0; j < KM; ++j)
    if (j < p.k) gd[j] = g[j];
  return bad;
}

// One CTA per tile; TPT > 0: the tile is exactly TPT sub-tiles and each
// thread keeps its TPT tokens' routes in registers from the histogram to the
// slot pass; TPT == 0: any number of sub-tiles, routes reloaded per pass.
// GATE: 0, or the fused gate for e <= GATE experts (8 or 32; router logits
// in; TPT > 0 only, since the routes stay in registers between the passes).
template <int TPT, int GATE, int KM>
__global__ void __launch_bounds__(kThreads) layout_kernel(const Params p) {
  static_assert(GATE == 0 || TPT > 0, "the fused gate keeps its routes in registers");
  constexpr int NM = TPT > 0 ? TPT : 1;
  __shared__ unsigned s_mask[NM][kWarps][kMaxE];
  __shared__ int s_wbase[NM][kWarps][kMaxE];
  __shared__ int s_agg[kMaxE];
  __shared__ int s_excl[kMaxE];
  __shared__ int s_tot[kMaxE];
  __shared__ int s_off[kMaxE + 1];
  __shared__ int s_rank[kMaxR];
  __shared__ int s_flags;  // bit 0: a bad route; 1: a wait timed out; 2: a non-finite logit; 3: rows exceeded
  __shared__ unsigned s_pub;  // this build's publish bit

  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int tile = blockIdx.x;
  const int nsub = (p.s + kThreads - 1) / kThreads;
  const int sub0 = tile * p.subtiles_per_tile;
  const int sub1 = min(nsub, sub0 + p.subtiles_per_tile);
  grid_dependency_wait();
  pdl_trigger_early();
  // the waits are bounded from here (not from the launch: a programmatic
  // launch may start this grid long before the previous kernel ends)
  const uint64_t deadline = globaltimer_ns() + (uint64_t)p.timeout_ns;
  if (p.e <= 32) {  // only the columns a route can touch
    for (int i = tid; i < NM * kWarps * 32; i += kThreads) (&s_mask[0][0][0])[(i >> 5) * kMaxE + (i & 31)] = 0u;
  } else {
    for (int i = tid; i < NM * kWarps * kMaxE; i += kThreads) (&s_mask[0][0][0])[i] = 0u;
  }
  for (int x = tid; x < kMaxE; x += kThreads) {
    s_agg[x] = 0;
    s_excl[x] = 0;
  }
  if (tid < kMaxR) s_rank[tid] = 0;
  // this tile's own row, as the previous build (or the zeroing) left it:
  // loaded now, used at the publication (its latency hides behind phase A)
  const unsigned own = tid == 0 ? ld_relaxed_u32(reinterpret_cast<const unsigned*>(p.out.lookback) +
                                                 (size_t)tile * padded_e(p.e))
                                : 0u;
  if (tid == 0) s_flags = 0;
  // a rebuild: tile 0 clears what the kernel accumulates into (published
  // with its look-back row, which every other tile reads before its atomics)
  if (p.clear_status && tile == 0) {
    if (tid == 0 && p.out.status) *p.out.status = 0;
    if (p.out.rank_counts && tid < p.R_tok) p.out.rank_counts[tid] = 0;
  }
  __syncthreads();

  // ---- A: token masks and the tile histogram -------------------------------
  int xs[NM][KM];
  unsigned valid[NM];
  bool bad = false;
  if (TPT > 0) {
#pragma unroll
    for (int r = 0; r < NM; ++r) {
      const int t = (sub0 + r) * kThreads + tid;
      valid[r] = 0;
      if (sub0 + r < sub1 && t < p.s) {
        if (GATE > 0) {
          if (gate_thread_token<KM, (GATE > 0 ? GATE : 8)>(p, t, xs[r])) atomicOr(&s_flags, 4);
          valid[r] = (1u << p.k) - 1u;  // k distinct ids in [0, e)
        } else {
          unsigned none;
          valid[r] = load_routes<KM>(p, t, xs[r], &none);
          bad |= (valid[r] | none) != (1u << p.k) - 1u;
        }
        store_route_ints<KM>(p.out.idx + unit_base(p, t), xs[r], p.k);
        mark_routes<KM>(p, s_mask[r], warp, lane, xs[r], valid[r]);
      }
    }
    __syncthreads();
    for (int x = tid; x < p.e; x += kThreads) {
      int run = 0;
#pragma unroll
      for (int r = 0; r < NM; ++r)
#pragma unroll
        for (int w = 0; w < kWarps; ++w) {
          s_wbase[r][w][x] = run;
          run += __popc(s_mask[r][w][x]);
        }
      s_agg[x] = run;
      s_tot[x] = run;
    }
  } else {
    for (int sb = sub0; sb < sub1; ++sb) {
      const int t = sb * kThreads + tid;
      int ys[KM];
      unsigned vy = 0;
      if (t < p.s) {
        unsigned none;
        vy = load_routes<KM>(p, t, ys, &none);
        bad |= (vy | none) != (1u << p.k) - 1u;
        store_route_ints<KM>(p.out.idx + unit_base(p, t), ys, p.k);
        mark_routes<KM>(p, s_mask[0], warp, lane, ys, vy);
      }
      __syncthreads();
      for (int x = tid; x < p.e; x += kThreads) {
        int c = 0;
#pragma unroll
        for (int w = 0; w < kWarps; ++w) c += __popc(s_mask[0][w][x]);
        s_agg[x] += c;
      }
      __syncthreads();
      for (int i = tid; i < kWarps * kMaxE; i += kThreads) (&s_mask[0][0][0])[i] = 0u;
      __syncthreads();
    }
    for (int x = tid; x < p.e; x += kThreads) s_tot[x] = s_agg[x];
  }
  if (bad) atomicOr(&s_flags, 1);
  if (tid == 0) s_pub = (own & kPublished) ? 0u : kPublished;
  __syncthreads();

  // ---- B: look-back over every earlier tile (all tiles when totals are needed)
  const bool last = tile == p.tiles - 1;
  const int nread = (p.capacity == 0 || last) ? p.tiles : tile;
  bool timed_out = false;
  lookback(p, tile, nread, s_agg, s_excl, s_tot, s_pub, deadline, &timed_out);
  if (timed_out) atomicOr(&s_flags, 2);
  // the look-back's shared atomics (none when it read no other tile)
  if (nread > (tile < nread ? 1 : 0)) __syncthreads();
  if (p.capacity == 0 || last) {
    expert_offsets(p, s_tot, s_off, last);
    __syncthreads();
  }

  // ---- C: token-order slots, rows, drops, dedup ----------------------------
  bool over = false;  // a route's row fell at or past the buffer's rows
  if (TPT > 0) {
#pragma unroll
    for (int r = 0; r < NM; ++r) {
      const int t = (sub0 + r) * kThreads + tid;
      unsigned long long ranks = 0;
      if (sub0 + r < sub1 && t < p.s)
        ranks = write_routes<KM>(p, t, lane, xs[r], valid[r], s_wbase[r][warp], s_excl, s_mask[r][warp], s_off,
                                 &over);
      if (p.R > 0) count_ranks(ranks, lane, s_rank);
    }
  } else {
    for (int x = tid; x < p.e; x += kThreads) s_agg[x] = s_excl[x];  // running base per expert
    __syncthreads();
    for (int sb = sub0; sb < sub1; ++sb) {
      const int t = sb * kThreads + tid;
      int ys[KM];
      unsigned vy = 0;
      if (t < p.s) {
        unsigned none;
        vy = load_routes<KM>(p, t, ys, &none);
        mark_routes<KM>(p, s_mask[0], warp, lane, ys, vy);
      }
      __syncthreads();
      for (int x = tid; x < p.e; x += kThreads) {
        int run = s_agg[x];
#pragma unroll
        for (int w = 0; w < kWarps; ++w) {
          s_wbase[0][w][x] = run;
          run += __popc(s_mask[0][w][x]);
        }
        s_agg[x] = run;
      }
      __syncthreads();
      unsigned long long ranks = 0;
      if (t < p.s)
        ranks = write_routes<KM>(p, t, lane, ys, vy, s_wbase[0][warp], nullptr, s_mask[0][warp], s_off, &over);
      if (p.R > 0) count_ranks(ranks, lane, s_rank);
      __syncthreads();
      for (int i = tid; i < kWarps * kMaxE; i += kThreads) (&s_mask[0][0][0])[i] = 0u;
      __syncthreads();
    }
  }
  if (over) atomicOr(&s_flags, 8);
  __syncthreads();
  pdl_trigger_late();
  // acquire, before an atomic on what tile 0 cleared in this build: word tid
  // of tile 0's published row, which tile 0's thread tid stored after
  // clearing rank_counts[tid] (and, for tid 0, the status word) and a fence.
  // The look-back already saw it published, so this load returns at once;
  // tile 0's own atomics follow its own clears.
  const bool rank_add = p.R > 0 && tid < p.R && s_rank[tid];
  if (tile != 0 && p.clear_status && (rank_add || (tid == 0 && s_flags)))
    (void)ld_acquire_u32(reinterpret_cast<const unsigned*>(p.out.lookback) + tid);
  if (rank_add) atomicAdd(&p.out.rank_counts[tid], s_rank[tid]);
  if (tid == 0 && s_flags) {
    int bits = 0;
    if (s_flags & 1) bits |= MOE_DEV_BAD_ROUTE;
    if (s_flags & 2) bits |= MOE_DEV_TIMEOUT;
    if (s_flags & 4) bits |= MOE_DEV_NONFINITE;
    if (s_flags & 8) bits |= MOE_DEV_ROWS_EXCEEDED;
    raise_status(p.out.status, bits);
  }
}

// k-major mode: the per-token work the unit scan cannot do -- expert ids
// repeated within a token, and the dedup rank sets -- from the rows the scan
// wrote.  One thread per token.
__global__ void __launch_bounds__(kThreads) token_ranks_kernel(const Params p) {
  __shared__ int s_rank[kMaxR];
  __shared__ int s_bad;
  const int tid = threadIdx.x, lane = tid & 31;
  grid_dependency_wait();
  if (tid < kMaxR) s_rank[tid] = 0;
  if (tid == 0) s_bad = 0;
  __syncthreads();
  const int per_rank = p.R_tok > 0 ? p.e / p.R_tok : 1;
  bool bad = false;
  for (int t0 = blockIdx.x * kThreads; t0 < p.s_tok; t0 += gridDim.x * kThreads) {
    const int t = t0 + tid;
    unsigned long long ranks = 0;
    if (t < p.s_tok) {
      int xs[kMaxK];
#pragma unroll
      for (int j = 0; j < kMaxK; ++j)
        if (j < p.k_tok) {
          xs[j] = __ldg(p.topk_idx + (size_t)t * p.k_tok + j);
          if (__ldg(p.out.row + (size_t)t * p.k_tok + j) >= 0) ranks |= 1ull << (xs[j] / per_rank);
#pragma unroll
          for (int jj = 0; jj < j; ++jj)
            if (xs[jj] == xs[j] && !(p.absent_ok && xs[j] == -1)) bad = true;
        }
      if (p.R_tok > 0) {
        uint8_t* tir = p.out.token_in_rank + (size_t)t * p.R_tok;
        for (int r = 0; r < p.R_tok; ++r) tir[r] = (uint8_t)((ranks >> r) & 1ull);
      }
    }
    if (p.R_tok > 0) count_ranks(ranks, lane, s_rank);
  }
  if (bad) atomicOr(&s_bad, 1);
  __syncthreads();
  if (p.R_tok > 0 && tid < p.R_tok && s_rank[tid]) atomicAdd(&p.out.rank_counts[tid], s_rank[tid]);
  if (tid == 0 && s_bad) raise_status(p.out.status, MOE_DEV_BAD_ROUTE);
}

int blocks_per_sm(const void* kern) {
  int n = 0;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, kern, kThreads, 0) != cudaSuccess) return 0;
  return n;
}

}  // namespace

LayoutPlan plan_layout(int s, int e, const DeviceInfo& di) {
  LayoutPlan plan;
  const int nsub = s > 0 ? (s + kThreads - 1) / kThreads : 1;
  int max_tiles = di.sms * (di.layout_blocks_per_sm > 0 ? di.layout_blocks_per_sm : 1);
  if (max_tiles > kMaxLookbackWords / padded_e(e)) max_tiles = kMaxLookbackWords / padded_e(e);
  plan.subtiles_per_tile = (nsub + max_tiles - 1) / max_tiles;
  if (plan.subtiles_per_tile < 1) plan.subtiles_per_tile = 1;
  plan.tiles = (nsub + plan.subtiles_per_tile - 1) / plan.subtiles_per_tile;
  if (plan.tiles < 1) plan.tiles = 1;
  return plan;
}

size_t lookback_bytes(const LayoutPlan& plan, int e) {
  return sizeof(unsigned) * (size_t)plan.tiles * (size_t)padded_e(e);
}

// The kernel variant of a sub-tile count (0 = any), a fused gate or not and
// the routes per unit rounded up to 1, 2, 4, 8 or 16.
template <int TPT, int GATE>
const void* layout_variant(int k) {
  if (k <= 1) return (const void*)layout_kernel<TPT, GATE, 1>;
  if (k <= 2) return (const void*)layout_kernel<TPT, GATE, 2>;
  if (k <= 4) return (const void*)layout_kernel<TPT, GATE, 4>;
  if (k <= 8) return (const void*)layout_kernel<TPT, GATE, 8>;
  return (const void*)layout_kernel<TPT, GATE, 16>;
}

int min_blocks(std::initializer_list<const void*> kerns) {
  int n = 1 << 30;
  for (const void* k : kerns) {
    const int b = blocks_per_sm(k);
    if (b < n) n = b;
  }
  return n;
}

// The fewest co-resident blocks per SM over the kernel variants, so that a
// plan fits whichever variant runs it.
int layout_blocks_per_sm() {
  int n = 1 << 30;
  for (int k : {1, 2, 4, 8, 16}) {
    const int b = min_blocks({layout_variant<0, 0>(k), layout_variant<1, 0>(k), layout_variant<2, 0>(k)});
    if (b < n) n = b;
  }
  return n;
}

// Co-resident CTAs per SM of the fused-gate variants.
int gate_layout_blocks_per_sm() {
  int n = 1 << 30;
  for (int k : {1, 2, 4, 8, 16}) {
    const int b = min_blocks({layout_variant<1, 8>(k), layout_variant<2, 8>(k), layout_variant<1, 32>(k),
                              layout_variant<2, 32>(k)});
    if (b < n) n = b;
  }
  return n;
}

std::atomic<bool> g_coop_pdl{true};  // the cooperative launch also takes programmatic serialisation

bool layout_can_fuse_gate(const LayoutPlan& plan, int priority, int e, const DeviceInfo& di) {
  return priority == 0 && e <= 32 && plan.subtiles_per_tile >= 1 && plan.subtiles_per_tile <= 2 &&
         plan.tiles <= di.sms * di.gate_layout_blocks_per_sm;
}

cudaError_t launch_layout(const int32_t* topk_idx, int s, int e, int k, int capacity, int R,
                          int priority, int pad_multiple, int rows, const LayoutPlan& plan,
                          const LayoutOut& out, int hold_tile, long long timeout_ns,
                          cudaStream_t st, const LayoutBuild& build) {
  Params p;
  p.topk_idx = topk_idx;
  p.kmajor = priority == 1;
  p.s = p.kmajor ? s * k : s;
  p.e = e;
  p.k = p.kmajor ? 1 : k;
  p.s_tok = s;
  p.k_tok = k;
  p.capacity = capacity;
  p.R = p.kmajor ? 0 : R;
  p.R_tok = R;
  p.pad = pad_multiple > 1 ? pad_multiple : 1;
  p.tiles = plan.tiles;
  p.subtiles_per_tile = plan.subtiles_per_tile;
  p.out = out;
  p.hold_tile = hold_tile;
  p.timeout_ns = timeout_ns;
  p.clear_status = build.clear_status;
  p.absent_ok = build.absent_ok;
  p.rows = rows;
  p.logits = build.logits;
  p.renorm = build.renorm;
  p.gate_idx = build.gate_idx;
  p.gate_val = build.gate_val;
  if (p.logits && (priority != 0 || e > 32 || plan.subtiles_per_tile < 1 || plan.subtiles_per_tile > 2))
    return cudaErrorInvalidValue;

  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(plan.tiles);
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = 0;
  cfg.stream = st;
  // cooperative (every tile co-resident), and with programmatic stream
  // serialisation where the driver takes both: the tiles may be scheduled
  // while the previous kernel drains; each waits for it (griddepcontrol.wait)
  // before its first read, and nothing that kernel runs waits on a tile.
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeCooperative;
  attr[0].val.cooperative = 1;
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[1].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = (MOE_PDL != 0 && ((MOE_PDL_MASK >> MOE_KERNEL_LAYOUT) & 1) && g_coop_pdl.load()) ? 2 : 1;
  cudaError_t err;
  const int tpt = plan.subtiles_per_tile;
  const void* kern = p.logits && e <= 8 ? (tpt == 1 ? layout_variant<1, 8>(p.k) : layout_variant<2, 8>(p.k))
                   : p.logits           ? (tpt == 1 ? layout_variant<1, 32>(p.k) : layout_variant<2, 32>(p.k))
                   : tpt == 1           ? layout_variant<1, 0>(p.k)
                   : tpt == 2           ? layout_variant<2, 0>(p.k)
                                        : layout_variant<0, 0>(p.k);
  void* args[] = {&p};
  err = cudaLaunchKernelExC(&cfg, kern, args);
  if (err != cudaSuccess && cfg.numAttrs == 2) {
    // the driver refused the pair of attributes: launch cooperative only,
    // from now on
    cudaGetLastError();
    g_coop_pdl.store(false);
    return launch_layout(topk_idx, s, e, k, capacity, R, priority, pad_multiple, rows, plan, out, hold_tile,
                         timeout_ns, st, build);
  }
  if (err != cudaSuccess || !p.kmajor || s == 0) return err;
  constexpr int kMaxPostBlocks = 1024;  // grid-stride beyond this
  int blocks = (s + kThreads - 1) / kThreads;
  if (blocks > kMaxPostBlocks) blocks = kMaxPostBlocks;
  token_ranks_kernel<<<blocks, kThreads, 0, st>>>(p);
  return cudaGetLastError();
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

// 64 KB: the tile plan never needs more than kMaxLookbackWords words; the
// launcher still refuses a plan that would not fit.
constexpr int kNoAllocLookbackWords = kMaxLookbackWords;

static __device__ __align__(256) unsigned g_noalloc_lookback[kNoAllocLookbackWords];

namespace {

struct NoAllocSetup {
  std::mutex mu;
  bool done = false;            // set only once every step below succeeded
  unsigned* scratch = nullptr;  // device address of g_noalloc_lookback
  DeviceInfo info;
};
NoAllocSetup g_noalloc[64];

// Per device, with that device current: resolve the scratch array's device
// address (its host-side name is only a stand-in) and the sizes the tile
// plan needs.  Allocates nothing.  A failure is returned and not latched, so
// a later call on the device tries again (a transient error, or a first call
// issued inside a stream capture, does not poison the device for good).
cudaError_t noalloc_setup(int dev, const NoAllocSetup** out) {
  NoAllocSetup& st = g_noalloc[dev];
  std::lock_guard<std::mutex> lk(st.mu);
  if (!st.done) {
    void* ptr = nullptr;
    cudaError_t err = cudaGetSymbolAddress(&ptr, g_noalloc_lookback);
    if (err != cudaSuccess) return err;
    DeviceInfo info;
    err = cudaDeviceGetAttribute(&info.sms, cudaDevAttrMultiProcessorCount, dev);
    if (err != cudaSuccess) return err;
    info.layout_blocks_per_sm = layout_blocks_per_sm();
    st.scratch = static_cast<unsigned*>(ptr);
    st.info = info;
    st.done = true;
  }
  *out = &st;
  return cudaSuccess;
}

}  // namespace

int noalloc_lookback_words() { return kNoAllocLookbackWords; }

cudaError_t launch_layout_noalloc(const int32_t* topk_idx, int s, int e, int k, int capacity, int R,
                                  const LayoutOut& out_in, int* words_needed, cudaStream_t st) {
  int dev = 0;
  cudaError_t err = cudaGetDevice(&dev);
  if (err != cudaSuccess) return err;
  if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  const NoAllocSetup* ps = nullptr;
  err = noalloc_setup(dev, &ps);
  if (err != cudaSuccess) return err;
  const NoAllocSetup& setup = *ps;

  const LayoutPlan plan = plan_layout(s, e, setup.info);
  const long long words = (long long)(lookback_bytes(plan, e) / sizeof(unsigned));
  *words_needed = (int)(words > 0x7fffffffLL ? 0x7fffffffLL : words);
  if (words > kNoAllocLookbackWords) return cudaErrorInvalidValue;  // caller reports the limit

  LayoutOut out = out_in;
  out.lookback = setup.scratch;
  err = cudaMemsetAsync(setup.scratch, 0, (size_t)words * sizeof(unsigned), st);
  if (err == cudaSuccess && R > 0)
    err = cudaMemsetAsync(out.rank_counts, 0, (size_t)R * sizeof(int32_t), st);
  if (err != cudaSuccess) return err;
  LayoutBuild build;  // status: the caller's word, OR-ed into
  const long long rows = capacity > 0 ? (long long)e * capacity : (long long)s * k;
  return launch_layout(topk_idx, s, e, k, capacity, R, 0, 1, (int)rows, plan, out, -1, 2000000000LL, st, build);
}

}  // namespace moe
