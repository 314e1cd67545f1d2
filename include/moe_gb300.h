/*
 * moe_gb300.h -- C ABI of the GB300 (sm_103a) mixture-of-experts token path:
 * top-k softmax gating, the dispatch layout, dispatch into the
 * expert-grouped buffer, the weighted combine, and the two backward duals
 * replayed on a cached layout handle; with them the router's gradient
 * (gate backward), layout variants (k-major capacity priority, per-expert
 * padding, per-virtual-rank send slots), the expert-grouped GEMM that
 * consumes the grouped rows (and its form fused with the dispatch), and an
 * allocation-free layout entry point.
 *
 * Sources (page title, then the part of the page that defines the call):
 *  [P1] NVIDIA-NeMo/Automodel #3684 "perf(moe): reuse the DeepEP dispatch
 *       layout on activation-checkpoint recompute": description and "How"
 *       (a handle from an earlier dispatch skips the layout; replayed
 *       counts must be identical to the forward's).
 *  [P3] deepspeedai/DeepSpeed #8213 "Add an opt-in DeepEP transport for the
 *       AutoEP expert all-to-all": description (a token is sent once per
 *       destination rank; the gradient of a combine is a dispatch and the
 *       gradient of a dispatch is a combine, both replayed on the forward's
 *       handle) and its review thread (the routing weights must really be
 *       applied in the combine; their gradient must reach the router; fp16
 *       is rejected; row counts come from the host, without a device read).
 *  [P4] deepspeedai/DeepSpeed #8195 "MoE dispatch: fix silent Tutel + TP
 *       corruption, speed up native and Tutel paths": change 1 (per-route
 *       index / location / gate, contiguous int32 routes, capacity resolved
 *       once), change 2 (the capacity buffer is [e, c, m], never a flat
 *       reinterpretation), change 3 (dispatch and combine are gathers
 *       through capacity slots; combine accumulates in fp32).
 *
 * Common rules
 *  - Every device pointer is caller-owned, device-resident on the current
 *    device, C-contiguous, 16-byte aligned, and is never retained after the
 *    call returns.  Tensor payload rows (m elements) must be a multiple of
 *    16 bytes long.
 *  - Every call only enqueues work on `stream` (a cudaStream_t passed as
 *    void*; NULL = the legacy default stream) and returns at once.  No call
 *    reads device memory on the host; row totals are host integers.
 *  - Arguments are validated on the host before anything is enqueued.  On
 *    any non-MOE_OK status nothing has been enqueued and no output changed.
 *  - Conditions only the device can see (non-finite logits, invalid expert
 *    ids, a bounded wait that ran out) set bits in a device status word; no
 *    kernel traps.  Read it with moe_handle_status (a synchronising helper).
 *  - Activations are fp32 or bf16; logits, gates and gate gradients fp32;
 *    expert ids and rows int32.  fp16 is rejected with MOE_ERR_DTYPE [P3].
 *  - Limits: 1 <= e <= 256, 1 <= k <= min(e, 16), 0 <= s, s*k < 2^31,
 *    rows < 2^31, 1 <= m, 0 <= R <= 64 with R dividing e.
 */
#ifndef MOE_GB300_H
#define MOE_GB300_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  MOE_OK = 0,
  MOE_ERR_INVALID_ARG = 1,     /* null / misaligned / out-of-range argument          */
  MOE_ERR_UNSUPPORTED = 2,     /* valid request this build does not support          */
  MOE_ERR_DTYPE = 3,           /* dtype other than fp32 / bf16 (fp16 included)       */
  MOE_ERR_HANDLE_MISMATCH = 4, /* handle unknown, destroyed, or sizes disagree      */
  MOE_ERR_CUDA = 5,            /* a CUDA runtime call failed                         */
  MOE_ERR_OOM = 6,             /* device allocation failed                           */
  MOE_ERR_TIMEOUT = 7,         /* device status: a bounded wait ran out              */
  MOE_ERR_NONFINITE = 8,       /* device status: a logit was NaN or infinite         */
  MOE_ERR_BAD_ROUTE = 9        /* device status: expert id out of range or repeated  */
} moe_status;

typedef enum { MOE_F32 = 0, MOE_BF16 = 1, MOE_F16 = 2 /* always rejected */ } moe_dtype;

/* Bits of a device status word (an int32 in device memory). */
#define MOE_DEV_NONFINITE 0x1
#define MOE_DEV_BAD_ROUTE 0x2
#define MOE_DEV_TIMEOUT 0x4
#define MOE_DEV_ROWS_EXCEEDED 0x8 /* dropless routes past the layout's rows_bound got no row */

/* Kernel ids for moe_launch_count. */
enum {
  MOE_KERNEL_TOPK_GATE = 0,
  MOE_KERNEL_LAYOUT = 1,
  MOE_KERNEL_DISPATCH = 2,
  MOE_KERNEL_COMBINE = 3,
  MOE_KERNEL_COMBINE_BWD = 4,
  MOE_KERNEL_DISPATCH_BWD = 5,
  MOE_KERNEL_TOPK_GATE_BWD = 6,
  MOE_KERNEL_GROUPED_GEMM = 7,
  MOE_KERNEL_DISPATCH_GEMM = 8,
  MOE_KERNEL_RANK_SLOTS = 9,
  MOE_KERNEL_COMBINE_GATE_BWD = 10,
  MOE_KERNEL_GATE_LAYOUT = 11,
  MOE_KERNEL_EP_PACK = 12,
  MOE_KERNEL_EP_UNPACK = 13,
  MOE_KERNEL_EP_DISPATCH = 14,
  MOE_KERNEL_EP_COMBINE = 15,
  MOE_KERNEL_COUNT = 16
};

/* Opaque layout handle [P1 "How"; P3 description].  Owned by the library:
 * built by moe_dispatch_layout, replayable any number of times by dispatch /
 * combine and their backwards, alive until moe_handle_destroy (so a backward
 * issued after later forwards still finds it).  Its device arrays come from a
 * library memory pool, allocated in stream order on the stream it was
 * created on and freed on the stream of its latest build.  A handle can also
 * be created empty (moe_layout_create) and built in place, again and again,
 * from new routes of the same shape (moe_layout_rebuild,
 * moe_topk_gate_layout): a build replaces the layout in stream order, so
 * work enqueued before it sees the old layout and work after it the new
 * one; builds of one handle must be ordered with each other and with every
 * use of the handle (one stream, or events). */
typedef struct moe_handle_s* moe_handle;

/* Capacity priority of moe_dispatch_layout_ex. */
enum {
  MOE_PRIORITY_TOKEN = 0,  /* slots fill in token order, each token's routes together */
  MOE_PRIORITY_KMAJOR = 1  /* every first choice before any second choice, ... */
};

/* Options of moe_dispatch_layout_ex. */
typedef struct {
  int32_t capacity;          /* slots per expert; 0 = dropless grouped layout        */
  int32_t num_virtual_ranks; /* dedup ranks R; 0 = none                              */
  int32_t priority;          /* MOE_PRIORITY_*                                       */
  int32_t pad_multiple;      /* dropless only: each expert's rows padded to a
                                multiple of this; 1 (or 0) = no padding            */
  int32_t send_slots;        /* 1: also build rank_slot (needs num_virtual_ranks > 0) */
  int32_t absent_routes;     /* 1: an expert id of -1 is a route that does not exist
                                (row -1, drop 1, no status bit): the layout of the
                                arrivals on an expert-parallel rank, whose routes to
                                other ranks are absent                             */
  int32_t rows_bound;        /* dropless without padding: the caller's bound on the
                                kept routes, used as the handle's rows instead of
                                s*k (e.g. an expert-parallel rank's route count,
                                known from the exchange of counts); 0 = s*k.  Routes
                                past it get no row (MOE_DEV_ROWS_EXCEEDED) and the
                                segments are cut there, so nothing reads or writes
                                past the rows                                       */
} moe_layout_options;

/* Host view of a handle: sizes and read-only device pointers. */
typedef struct {
  int32_t s, e, k;
  int32_t capacity;   /* slots per expert; 0 = dropless grouped layout          */
  int32_t R;          /* virtual ranks of the dedup counts; 0 = none            */
  int32_t rows;       /* rows of the dispatched buffer: e*capacity, or s*k      */
  int32_t device;     /* CUDA device the handle lives on                        */
  int32_t priority;   /* MOE_PRIORITY_TOKEN or MOE_PRIORITY_KMAJOR               */
  int32_t pad_multiple; /* dropless segments padded to a multiple of this (>= 1) */
  const int32_t* idx;           /* [s,k] copy of the expert ids                 */
  const int32_t* loc;           /* [s,k] token-order slot within the expert     */
  const int32_t* row;           /* [s,k] row in the dispatched buffer, -1 = dropped */
  const uint8_t* drop;          /* [s,k] 1 = dropped (capacity) or invalid      */
  const int32_t* raw_counts;    /* [e]   routes per expert before capacity      */
  const int32_t* counts;        /* [e]   kept routes per expert                 */
  const int32_t* offsets;       /* [e+1] first row of each expert; [e] = rows   */
  const uint8_t* token_in_rank; /* [s,R] 1 = token sends to that virtual rank   */
  const int32_t* rank_counts;   /* [R]   tokens sent to each virtual rank       */
  const int32_t* status;        /* device status word of this handle            */
  const int32_t* inv_row;       /* [rows] token whose kept route owns the row;
                                   unspecified at rows no route owns           */
  const int32_t* rank_slot;     /* [s,R] token-order send slot per virtual rank,
                                   -1 = not sent; NULL unless send_slots = 1   */
} moe_layout_info;

/* Top-k softmax gating [P4 change 1; P1 description: recompute must route
 * identically].  logits f32 [s,e] -> topk_idx i32 [s,k], topk_gate f32 [s,k].
 * Selection is on the logits: larger first, the lower expert index on ties
 * (+0.0 and -0.0 tie).  renorm = 0: gate = softmax over all e experts, read
 * at the selected ones; renorm = 1: softmax over the k selected logits.
 * fp32 arithmetic with expf.  Deterministic.  device_status (nullable): an
 * int32 in device memory that gets MOE_DEV_NONFINITE OR-ed in when a logit
 * of a token is NaN or infinite (that token's outputs are then unspecified).
 */
moe_status moe_topk_gate(const float* logits, int s, int e, int k, int renorm,
                         int32_t* topk_idx, float* topk_gate, int32_t* device_status,
                         void* stream);

/* Top-k gate backward [P3 review thread: the routing weights' gradient must
 * reach the router gate, or the router silently never learns].  With the
 * selection held fixed (top-k is piecewise constant in the logits):
 *   renorm = 1: dlogits[i_j] = g_j * (dgate_j - sum_j' g_j' * dgate_j'),
 *               every other expert 0;
 *   renorm = 0: dlogits[i] = p_i * (dgate(i) - sum_j g_j * dgate_j), p the
 *               softmax of the logits over all e experts (recomputed here in
 *               fp32 with expf), dgate(i) = dgate_j for i = i_j, else 0.
 * logits f32 [s,e] (may be NULL when renorm = 1), topk_idx i32 [s,k] and
 * topk_gate f32 [s,k] as returned by moe_topk_gate, dgate f32 [s,k]
 * (e.g. from moe_combine_bwd) -> dlogits f32 [s,e].  fp32 arithmetic, fixed
 * summation order.  Expert ids must be in [0, e) and distinct per token. */
moe_status moe_topk_gate_bwd(const float* logits, const int32_t* topk_idx, const float* topk_gate,
                             const float* dgate, int s, int e, int k, int renorm, float* dlogits,
                             void* stream);

/* Dispatch layout [P4 changes 1 and 3: location = cumulative count - 1 in
 * token order; P3 description: dedup once per destination rank].
 * topk_idx i32 [s,k] -> a new handle in *out (see moe_layout_info):
 *   loc[t,j]  = number of earlier tokens t' < t routed to expert idx[t,j];
 *   capacity > 0: dropped iff loc >= capacity; row = x*capacity + loc;
 *                 counts = min(raw_counts, capacity); offsets[x] = x*capacity;
 *   capacity = 0: nothing dropped; offsets = exclusive prefix of counts;
 *                 row = offsets[x] + loc;
 *   R > 0: token_in_rank[t,r] = 1 iff a kept route of t goes to one of the
 *          e/R experts of virtual rank r; rank_counts[r] = sum over t.
 *          Computed only; nothing is sent anywhere.
 * One kernel: a shared-memory histogram per tile and a decoupled look-back
 * over tiles; integer-exact and bitwise reproducible on every rebuild.
 * Expert ids out of [0, e) or repeated within a token are reported through
 * the handle's status word (MOE_DEV_BAD_ROUTE) and those routes get
 * row = -1.  Errors: MOE_ERR_INVALID_ARG, MOE_ERR_OOM, MOE_ERR_CUDA. */
moe_status moe_dispatch_layout(const int32_t* topk_idx, int s, int e, int k, int capacity,
                               int num_virtual_ranks, void* stream, moe_handle* out);

/* An empty layout handle for s tokens, e experts, k routes per token and the
 * layout options of moe_dispatch_layout_ex: its device arrays are allocated
 * (and their flags zeroed) on `stream`, but it holds no layout until the
 * first moe_layout_rebuild or moe_topk_gate_layout; payload calls on it
 * before that return MOE_ERR_INVALID_ARG.  For per-step builds that should
 * not allocate [P1 description: the layout is recomputed every step].
 * Errors as moe_dispatch_layout_ex. */
moe_status moe_layout_create(int s, int e, int k, const moe_layout_options* options, void* stream,
                             moe_handle* out);

/* Build (or rebuild) h's layout in place from new expert ids topk_idx
 * i32 [h.s, h.k]: the same arrays, counts and status as
 * moe_dispatch_layout_ex with h's options would give, written into h's own
 * memory with no allocation and no memset (the layout kernel clears the
 * status word and rank counts itself).  See moe_handle on ordering.
 * Errors: MOE_ERR_INVALID_ARG, MOE_ERR_HANDLE_MISMATCH, MOE_ERR_CUDA. */
moe_status moe_layout_rebuild(moe_handle h, const int32_t* topk_idx, void* stream);

/* Top-k gating fused into the layout build [P4 change 1; P1 description].
 * logits f32 [h.s, h.e] -> topk_idx i32 [h.s, h.k] and topk_gate f32
 * [h.s, h.k] exactly as moe_topk_gate(logits, ..., renorm) writes them, and
 * h's layout built from those ids as moe_layout_rebuild would.  With up to
 * 32 experts (token priority, batches whose layout tiles span at most two
 * sub-tiles of 256 tokens) this is one kernel, in which each token's thread
 * selects its experts before the tile counts them; otherwise it is the gate
 * kernel followed by the layout kernel (measured faster there than a fused
 * form), with the same results.  No allocation and no memset either way.
 * Non-finite logits set MOE_DEV_NONFINITE in h's status word.  Errors as
 * moe_layout_rebuild; renorm other than 0 or 1 is MOE_ERR_INVALID_ARG. */
moe_status moe_topk_gate_layout(moe_handle h, const float* logits, int renorm, int32_t* topk_idx,
                                float* topk_gate, void* stream);

/* Allocation-free dispatch layout.  The paper has no counterpart: an
 * addition of this library for callers that cannot allocate device memory
 * when they build a layout (inside a captured CUDA graph where a pool
 * allocation is unwanted, from an allocator's own hook that must not
 * re-enter it, or in runtimes that hand out only fixed buffers).
 * Computes exactly what moe_dispatch_layout computes, but writes it into
 * caller-owned arrays instead of a handle: idx_out, loc, row [s,k] int32;
 * drop [s,k] uint8; raw_counts, counts [e] int32; offsets [e+1] int32; and,
 * when num_virtual_ranks R > 0, token_in_rank [s,R] uint8 and rank_counts
 * [R] int32 (ignored when R = 0).  device_status (nullable): an int32 in
 * device memory that gets MOE_DEV_* bits OR-ed in (the caller zeroes it).
 * It calls no allocating routine.  The kernel's scratch (its look-back
 * words: tiles x (e rounded up to a multiple of 4) of them) is a fixed
 * library array of 16384 32-bit words (64 KB) per device, held until the
 * process exits.  The tile plan keeps that product within 16384 for every
 * accepted size; a plan that would need more returns
 * MOE_ERR_UNSUPPORTED (use moe_dispatch_layout) instead of overrunning it.  Every call shares
 * that array and clears the part it uses, so calls whose work overlaps on the
 * GPU (unordered streams) race; order them.  The first call on each device
 * resolves the array's device address (one-time set-up); make that first call
 * before any stream capture.  A set-up that fails is not remembered: the
 * call returns the error and the next call on that device tries again.  The dispatch / combine calls still take a
 * handle, so this suits callers that consume the layout arrays themselves. */
moe_status moe_dispatch_layout_noalloc(const int32_t* topk_idx, int s, int e, int k, int capacity,
                                       int num_virtual_ranks, int32_t* idx_out, int32_t* loc,
                                       int32_t* row, uint8_t* drop, int32_t* raw_counts,
                                       int32_t* counts, int32_t* offsets, uint8_t* token_in_rank,
                                       int32_t* rank_counts, int32_t* device_status, void* stream);

/* Dispatch layout with options [P4 change 1: the routes' capacity ranking;
 * Automodel #3684 description: per-expert padding of the grouped rows].
 * As moe_dispatch_layout, plus:
 *   priority = MOE_PRIORITY_KMAJOR: loc[t,j] counts the routes to the same
 *     expert with j' < j, or j' == j and t' < t (GShard's order: a first
 *     choice is never dropped for a later choice of another token);
 *   pad_multiple = P > 1 (dropless only): offsets[x+1] = offsets[x] +
 *     ceil(counts[x] / P) * P; the handle's rows is the upper bound
 *     s*k + e*(P-1), so it stays a host integer; dispatch and the combine
 *     backward write zeros into padding rows and rows past offsets[e];
 *   send_slots = 1 (needs num_virtual_ranks R > 0) [DeepSpeed #8213
 *     description: a token goes to a destination rank once]: rank_slot
 *     [s,R] int32, rank_slot[t,r] = #{t' < t : token_in_rank[t',r]} where
 *     token_in_rank[t,r] = 1, else -1: each token's slot in the send buffer
 *     of every virtual rank it goes to, in token order (whatever the
 *     capacity priority); rank r's slots are 0 .. rank_counts[r]-1.  One more
 *     kernel (MOE_KERNEL_RANK_SLOTS), one CTA per rank.
 * Errors as moe_dispatch_layout; pad_multiple > 1 with capacity > 0, an
 * unknown priority, or send_slots without virtual ranks is
 * MOE_ERR_INVALID_ARG. */
moe_status moe_dispatch_layout_ex(const int32_t* topk_idx, int s, int e, int k,
                                  const moe_layout_options* options, void* stream, moe_handle* out);

/* Dispatch [P4 change 3; P4 change 2 for the [e, c, m] layout].
 * x [s,m] -> X [rows,m]: X[row[t,j]] = x[t] for every kept route; in
 * capacity mode the unused slots [counts[x], capacity) of every expert are
 * written with zeros, so X is fully defined.  Bit-exact copy.
 * s and rows must equal the handle's (else MOE_ERR_HANDLE_MISMATCH). */
moe_status moe_dispatch(moe_handle h, int s, int rows, int m, moe_dtype dtype,
                        const void* x, void* X, void* stream);

/* Combine [P3 review thread: the weights are applied; P4 change 3: fp32
 * accumulation].  y [rows,m], gate f32 [s,k] -> out [s,m]:
 *   acc = +0.0f; for j = 0..k-1 with row[t,j] >= 0:
 *       acc = fmaf(gate[t,j], (float)y[row[t,j]], acc);
 *   out[t] = acc rounded to nearest-even in the output type.
 * A token whose routes were all dropped gets zeros.  gate may not be NULL. */
moe_status moe_combine(moe_handle h, int s, int rows, int m, moe_dtype dtype,
                       const void* y, const float* gate, void* out, void* stream);

/* Combine backward = a dispatch [P3 description].  dout [s,m], gate f32
 * [s,k], y [rows,m] -> dY [rows,m], dgate f32 [s,k]:
 *   dY[row[t,j]] = (gate[t,j] * (float)dout[t]) rounded to the type (one fp32
 *   multiply, then nearest-even); rows no kept route owns are zero;
 *   dgate[t,j] = sum_m dout[t,m]*y[row[t,j],m] accumulated in fp32; 0 if the
 *   route was dropped.  This is the router's gradient path [P3 review]. */
moe_status moe_combine_bwd(moe_handle h, int s, int rows, int m, moe_dtype dtype,
                           const void* dout, const float* gate, const void* y,
                           void* dY, float* dgate, void* stream);

/* Combine backward with the top-k gate backward fused in [P3 description:
 * combine-grad = dispatch; P3 review thread: the routing weights' gradient
 * must reach the router].  Exactly moe_combine_bwd followed by
 * moe_topk_gate_bwd(logits, idx, gate, dgate, ...) on the handle's own
 * expert ids (its idx copy), in one kernel: dY [rows,m] and dgate f32 [s,k]
 * as moe_combine_bwd, and dlogits f32 [s,e] as moe_topk_gate_bwd -- the same
 * bits as the two calls.  Each token's router gradient is written by the
 * warp that reduced its gate gradients, so dgate is never re-read.
 * logits f32 [s,e] is read only when renorm = 0 (may be NULL when renorm =
 * 1).  Errors as moe_combine_bwd; renorm other than 0 or 1 is
 * MOE_ERR_INVALID_ARG. */
moe_status moe_combine_gate_bwd(moe_handle h, int s, int rows, int m, moe_dtype dtype,
                                const void* dout, const float* gate, const void* y,
                                const float* logits, int renorm, void* dY, float* dgate,
                                float* dlogits, void* stream);

/* Dispatch backward = a combine with unit weights [P3 description].
 * dX [rows,m] -> dx [s,m]: dx[t] = sum over kept routes, in route order,
 * accumulated in fp32 as in moe_combine. */
moe_status moe_dispatch_bwd(moe_handle h, int s, int rows, int m, moe_dtype dtype,
                            const void* dX, void* dx, void* stream);

/* ---- Expert-parallel exchange [P3 description: a token goes to each
 * destination rank once, not once per selected expert; the transport
 * replicates it, groups the arrivals by expert and reduces in its combine;
 * P3 review thread: the routing weights travel with the tokens and are
 * applied on the expert's rank, their gradient returns to the router].
 * Rank r of R owns experts [r*E, (r+1)*E), E = e/R.  On the source rank,
 * h is the layout of its routes built with num_virtual_ranks = R and
 * send_slots = 1 (1 <= R <= 32).  The send buffer holds R destination
 * segments in rank order, segment r = the tokens with a kept route to rank
 * r in token order, rows_sent = sum of h's rank_counts (a host integer the
 * caller obtains once per layout, e.g. with the all-to-all of the counts
 * that sizes the exchange).  The all-to-all itself is the caller's (NCCL);
 * these calls are the per-rank steps around it.  On the destination, the
 * arrivals (segments from source 0, 1, ...) get their own layout from the
 * received meta_idx with absent_routes = 1 and go through moe_dispatch /
 * moe_combine(gate = the received meta_gate) / their backwards as any
 * batch does; each arrival's combined row is its partial, sent back.
 * Errors: MOE_ERR_INVALID_ARG (no send slots, R outside [1, 32], sizes,
 * pointers), MOE_ERR_HANDLE_MISMATCH, MOE_ERR_CUDA. */

/* send_row i32 [s,R]: send_row[t,r] = the row of token t in the send
 * buffer's segment r, or -1; and, per sent row q, the token's k routes as
 * the destination sees them: meta_idx i32 [rows_sent,k] = local expert id
 * (idx - r*E) of a kept route to rank r, else -1; meta_gate f32
 * [rows_sent,k] = its gate, else 0.  A send slot at or past rows_sent is
 * not sent and sets MOE_DEV_BAD_ROUTE in h's status word. */
moe_status moe_ep_pack(moe_handle h, const float* gate, int rows_sent, int32_t* send_row,
                       int32_t* meta_idx, float* meta_gate, void* stream);

/* The send buffer: X_send[send_row[t,r]] = x[t] for every r with
 * send_row[t,r] >= 0 -- each token row read once, written once per
 * destination rank (the dispatch kernel over the send map).  x [s,m],
 * X_send [rows_sent,m]; rows at or past rows_sent are never written. */
moe_status moe_ep_dispatch(moe_handle h, const int32_t* send_row, int rows_sent, int m, moe_dtype dtype,
                           const void* x, void* X_send, void* stream);

/* The source's reduction of the partials that came back (P [rows_sent,m],
 * each at the row its token was sent from): out[t] = sum over r in rank
 * order of P[send_row[t,r]], accumulated in fp32 and rounded once; a token
 * that sent nothing gets zeros.  Also the backward of moe_ep_dispatch
 * (dx from the returned gradients). */
moe_status moe_ep_combine(moe_handle h, const int32_t* send_row, int rows_sent, int m, moe_dtype dtype,
                          const void* P, void* out, void* stream);

/* The gate gradients that came back (dgate_back f32 [rows_sent,k], row q =
 * the destination's gradients of the sent token's k routes) to the
 * source's routes: dgate[t,j] = dgate_back[send_row[t, idx[t,j]/E], j] for
 * a kept route, 0 for a dropped one. */
moe_status moe_ep_unpack_dgate(moe_handle h, const int32_t* send_row, int rows_sent, const float* dgate_back,
                               float* dgate, void* stream);

/* Expert-grouped GEMM over the dispatched buffer, on the tensor cores
 * [P3 description: the dispatch groups arrivals by expert for the grouped
 * GEMM, groups bounded by offsets = cumsum(counts)].  For every row r that a
 * kept route to expert x owns, r in [offsets[x], offsets[x] + counts[x]):
 *   Y[r, :] = X[r, :] . W[x]^T   (bf16 in, fp32 accumulation, bf16 out,
 *                                 round to nearest-even)
 * X bf16 [rows, K] (the output of moe_dispatch), W bf16 [e, N, K] (each
 * expert's weight N x K with K contiguous), Y bf16 [rows, N].  Rows no route
 * owns (capacity tails, padding) are not written.  Any layout of the handle:
 * token or k-major, capacity or dropless, padded or not.  K a multiple of
 * 8 and at least 64; N a multiple of 8 (16-byte rows); rows equal to the
 * handle's; e <= 256.
 * tcgen05 MMA on pairs of SMs (cta_group::2) with TMEM accumulators,
 * TMA-fed; the segments are read from the handle on the device (no host
 * sync).  Errors: MOE_ERR_INVALID_ARG, MOE_ERR_HANDLE_MISMATCH,
 * MOE_ERR_CUDA. */
moe_status moe_grouped_gemm(moe_handle h, int rows, int K, int N, const void* X, const void* W,
                            void* Y, void* stream);

/* Dispatch fused into the grouped GEMM [P3 description: the grouped GEMM
 * consumes the arrivals grouped by expert; P4 change 3: gather rows by index
 * instead of materialising a one-hot product].  The same Y as
 * moe_dispatch followed by moe_grouped_gemm, without the dispatched buffer:
 * the A operand's rows are gathered from the token rows through the
 * handle's inv_row (row -> token), straight into the GEMM's shared-memory
 * tiles.
 *   Y[r, :] = x[inv_row[r], :] . W[x]^T   for every owned row r,
 * x bf16 [s, K] (the tokens' activations, K = m), W bf16 [e, N, K], Y bf16
 * [rows, N]; rows no route owns are not written.  Each owned row equals
 * moe_grouped_gemm's bit for bit (same operands, same MMA sequence).  Same
 * limits and errors as moe_grouped_gemm; s must equal the handle's.
 * Each token row is gathered once per 256-column tile of N, mostly from L2
 * (the column tiles of a row block run on different SM pairs at the same
 * time): on every measured shape the fused call beat moe_dispatch followed
 * by moe_grouped_gemm, by 3 % (16384 tokens of 4096, N = 4096) to 26 %
 * (the GShard-like capacity layout). */
moe_status moe_dispatch_grouped_gemm(moe_handle h, int s, int rows, int K, int N, const void* x,
                                     const void* W, void* Y, void* stream);

/* Fill *info with the handle's sizes and device pointers (valid until the
 * handle is destroyed). */
moe_status moe_handle_info(moe_handle h, moe_layout_info* info);

/* Synchronise `stream`, then copy the handle's device status word (bits
 * MOE_DEV_*) to *device_status.  A test / debugging helper: it blocks. */
moe_status moe_handle_status(moe_handle h, void* stream, int32_t* device_status);

/* Release the handle: its device arrays are freed in stream order on the
 * stream it was built on, so work already enqueued there that uses it
 * completes first.  Work on other streams must be complete (or ordered
 * before that stream) by the caller.  Using the handle afterwards returns
 * MOE_ERR_HANDLE_MISMATCH. */
moe_status moe_handle_destroy(moe_handle h);

/* ceil(capacity_factor * s * k / e) computed in double on the host
 * [P4 change 1: capacity resolved once]; 0 if an argument is out of range. */
int moe_capacity(double capacity_factor, int s, int k, int e);

/* Static text for a status code. */
const char* moe_status_string(moe_status st);

/* Text of the last validation or CUDA error seen by this host thread. */
const char* moe_last_error(void);

/* Number of launches of one kernel (MOE_KERNEL_*) since the library was
 * loaded, process-wide.  A replay on a cached handle leaves the layout
 * count unchanged [P1 "How"]. */
uint64_t moe_launch_count(int kernel_id);

/* Test hook for the bounded waits: the next layout build whose tile count
 * exceeds `tile` leaves that tile's look-back words unpublished for twice
 * timeout_ms, so every tile that waits on it gives up (after timeout_ms) and
 * sets MOE_DEV_TIMEOUT in the handle's status word.  The hook disarms itself after one build;
 * tile = -1 disarms it.  Never used on the product path. */
moe_status moe_debug_hold_layout_tile(int tile, int timeout_ms);

#ifdef __cplusplus
}
#endif
#endif /* MOE_GB300_H */
