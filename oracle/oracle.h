/*
 * oracle.h -- plain, slow, obviously-correct CPU implementation of the MoE
 * token path (top-k softmax gating, dispatch layout, dispatch, combine and
 * their backward duals).
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing on the product path may link, load or
 * call this code: only the test-suite, the smoke check and the CPU-baseline
 * leg of the benchmark do.  It shares no header, helper, table or constant
 * with the CUDA library; its enums and its bf16 conversion are its own.
 *
 * Sources the definitions follow (page title, then the part of the page):
 *  [P1] NVIDIA-NeMo/Automodel #3684 "perf(moe): reuse the DeepEP dispatch
 *       layout on activation-checkpoint recompute" -- description, "How".
 *  [P3] deepspeedai/DeepSpeed #8213 "Add an opt-in DeepEP transport for the
 *       AutoEP expert all-to-all" -- description (dedup, duality) and the
 *       review thread on weighted combine.
 *  [P4] deepspeedai/DeepSpeed #8195 "MoE dispatch: fix silent Tutel + TP
 *       corruption, speed up native and Tutel paths" -- changes 1 and 3.
 *
 * Conventions: row-major C arrays; s tokens, e experts, k routes per token,
 * m hidden size; a "route" is (t, j) with j in [0, k).  bf16 tensors are
 * passed as raw uint16 bit patterns.  Every function returns 0 on success
 * and a negative ORA_E* code on a contract violation (it then leaves the
 * outputs unspecified).  No function allocates memory it does not free.
 *
 * Threading: the per-token loops of gate / dispatch / combine / backward may
 * be split across OpenMP threads (ora_set_threads); every output element is
 * written by exactly one thread with the same arithmetic, so results do not
 * depend on the thread count.  The layout scan is sequential.
 */
#ifndef MOE_ORACLE_H
#define MOE_ORACLE_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

enum { ORA_F32 = 0, ORA_BF16 = 1 };

enum {
  ORA_OK = 0,
  ORA_EARG = -1,      /* sizes out of range, null pointer            */
  ORA_ENONFINITE = -2,/* a logit is NaN or +-inf                     */
  ORA_EROUTE = -3     /* expert id out of range, or repeated in a token */
};

/* Number of OpenMP threads the per-token loops use (>= 1).  Returns the
 * count actually in effect (1 when built without OpenMP). */
int ora_set_threads(int n);
int ora_get_threads(void);

/* bf16 <-> f32.  Widening is exact; narrowing rounds to nearest, ties to
 * even, and keeps NaN a (quiet) NaN. */
float ora_bf16_to_f32(uint16_t b);
uint16_t ora_f32_to_bf16(float f);

/* Top-k softmax gating [P4 change 1; P1 description].
 * logits f32 [s,e]  ->  idx i32 [s,k], gate f32 [s,k].
 * Selection on the logits: expert j gets position
 *   pos(j) = #{ i : l_i > l_j  or  (l_i == l_j and i < j) }
 * and is selected iff pos(j) < k (larger logit first, lower index on ties).
 * renorm = 0: gate = exp(l_j - M) / sum_{i<e} exp(l_i - M), M = max_i l_i.
 * renorm = 1: the same ratio over the k selected experts only.
 * Computed in double, rounded once to float. */
int ora_topk_gate(const float* logits, int s, int e, int k, int renorm,
                  int32_t* idx, float* gate);

/* Top-k gate backward [P3 review thread: the routing weights' gradient must
 * reach the router].  With the selection idx fixed (it is piecewise
 * constant in the logits), the gates are a softmax of the logits:
 * renorm = 1: g_j = exp(l_{i_j}) / sum_{j'} exp(l_{i_j'}) over the selected;
 *   dlogits[i_j] = g_j * (dgate_j - sum_{j'} g_{j'} dgate_{j'}), others 0.
 * renorm = 0: g_j = p_{i_j}, p = softmax over all e logits;
 *   dlogits[i] = p_i * (dgate(i) - sum_j g_j dgate_j), dgate(i) = dgate_j
 *   when i = i_j, else 0 (every expert gets a gradient).
 * gate holds the forward's gates; p is recomputed from the logits in double.
 * Everything in double, rounded once to float. */
int ora_topk_gate_bwd(const float* logits, const int32_t* idx, const float* gate,
                      const float* dgate, int s, int e, int k, int renorm, float* dlogits);

/* Dispatch layout [P4 change 1 and 3: location = cumsum - 1 in token order;
 * P3 description: one send per destination rank].
 * loc[t,j]  = #{ t' < t : expert idx[t,j] is among idx[t',:] }
 * raw_counts[x] = number of routes to x.
 * capacity > 0: drop = loc >= capacity; counts = min(raw, capacity);
 *               row = x*capacity + loc (or -1 if dropped);
 *               offsets[x] = x*capacity (x in [0, e]).
 * capacity = 0: nothing dropped; counts = raw;
 *               offsets = exclusive prefix sum of counts (offsets[e] = s*k);
 *               row = offsets[x] + loc.
 * R > 0 (R divides e, experts grouped e/R per virtual rank):
 *   token_in_rank[t,r] = 1 iff some kept route of t goes to an expert of r;
 *   rank_counts[r] = sum_t token_in_rank[t,r].
 * token_in_rank / rank_counts may be NULL when R = 0. */
int ora_layout(const int32_t* idx, int s, int e, int k, int capacity, int R,
               int32_t* loc, int32_t* row, uint8_t* drop,
               int32_t* raw_counts, int32_t* counts, int32_t* offsets,
               uint8_t* token_in_rank, int32_t* rank_counts);

/* Layout variants [P4 change 1: routes ranked for capacity; Automodel #3684
 * description: HybridEP pads each expert's rows to pad_multiple].
 * priority = 0: token order (ora_layout).  priority = 1: k-major (all first
 *   choices before any second choice): loc[t,j] = #{ (t',j') routed to the
 *   same expert with j' < j, or j' == j and t' < t }.
 * pad_multiple = P >= 1 (dropless only): each expert's rows are padded to a
 *   multiple of P: offsets[x+1] = offsets[x] + ceil(counts[x] / P) * P, and
 *   `rows` = s*k + e*(P-1) is the buffer size the caller allocates (an upper
 *   bound of offsets[e]).  P = 1 is the plain grouped layout.
 * Dedup and drops as in ora_layout (drops apply to the k-major locations). */
int ora_layout_ex(const int32_t* idx, int s, int e, int k, int capacity, int R, int priority,
                  int pad_multiple, int32_t* loc, int32_t* row, uint8_t* drop,
                  int32_t* raw_counts, int32_t* counts, int32_t* offsets,
                  uint8_t* token_in_rank, int32_t* rank_counts);

/* Per-virtual-rank send slots [DeepSpeed #8213 description: a token goes to
 * each destination rank once, whatever number of that rank's experts it
 * selected].  For every rank r, the tokens that send to r (token_in_rank
 * [s,R] from ora_layout) are numbered in token order:
 *   rank_slot[t,r] = #{ t' < t : token_in_rank[t',r] = 1 }  if token_in_rank[t,r]
 *                  = -1                                     otherwise,
 * so slot values of rank r run 0 .. rank_counts[r]-1. */
int ora_rank_slots(const uint8_t* token_in_rank, int s, int R, int32_t* rank_slot);

/* Dispatch [P4 change 3]: X has `rows` rows of m elements; every row is first
 * zero, then X[row[t,j]] = x[t] for each kept route (row >= 0). */
int ora_dispatch(const int32_t* row, int s, int k, int m, int dtype,
                 const void* x, int rows, void* X);

/* Combine [P3 review thread: the routing weights must be applied; P4
 * change 3: accumulate in fp32]:
 *   acc = 0.0f; for j = 0..k-1, if row[t,j] >= 0:
 *       acc = fmaf(gate[t,j], (float)y[row[t,j]], acc);
 *   out[t] = acc rounded to the output type.
 * gate == NULL means unit weights (this is dispatch's backward). */
int ora_combine(const int32_t* row, const float* gate, int s, int k, int m,
                int dtype, const void* y, void* out);

/* Combine backward [P3 description: the gradient of a combine is a dispatch]:
 *   dY[row[t,j]] = (gate[t,j] * (float)dout[t]) rounded to the type
 *                  (the product is one fp32 multiply), other rows zero;
 *   dgate[t,j]   = sum_m (double)dout[t,m] * (double)y[row[t,j],m],
 *                  rounded to float; 0 for a dropped route. */
int ora_combine_bwd(const int32_t* row, const float* gate, int s, int k, int m,
                    int dtype, const void* dout, const void* y, int rows,
                    void* dY, float* dgate);

/* Dispatch backward [P3 description: the gradient of a dispatch is a
 * combine]: ora_combine with unit weights. */
int ora_dispatch_bwd(const int32_t* row, int s, int k, int m, int dtype,
                     const void* dX, void* dx);

#ifdef __cplusplus
}
#endif
#endif
