/*
 * oracle.c -- the CPU oracle for the MoE token path.  TEST INFRASTRUCTURE
 * ONLY: see oracle.h for the definitions, their sources and the rules on
 * who may call this file.
 *
 * Written for readability, not speed: each function is the plain definition
 * from oracle.h in the order stated there.  Compile with
 * -ffp-contract=off so that no a*b+c is silently fused (the only fused
 * multiply-add is the explicit fmaf of the combine).
 */
#include "oracle.h"

#include <math.h>
#include <stddef.h>
#include <stdlib.h>
#include <string.h>

#ifdef _OPENMP
#include <omp.h>
#endif

static int g_threads = 1;

int ora_set_threads(int n) {
#ifdef _OPENMP
  g_threads = n < 1 ? 1 : n;
#else
  (void)n;
  g_threads = 1;
#endif
  return g_threads;
}

int ora_get_threads(void) { return g_threads; }

/* ---------------------------------------------------------------- bf16 -- */

float ora_bf16_to_f32(uint16_t b) {
  uint32_t u = (uint32_t)b << 16;
  float f;
  memcpy(&f, &u, sizeof f);
  return f;
}

uint16_t ora_f32_to_bf16(float f) {
  uint32_t u;
  memcpy(&u, &f, sizeof u);
  if ((u & 0x7f800000u) == 0x7f800000u && (u & 0x007fffffu) != 0) {
    /* NaN: keep the sign, force a quiet NaN */
    return (uint16_t)((u >> 16) | 0x0040u);
  }
  /* Keep the upper 16 bits, rounding the lower 16 to nearest, ties to even:
   * add 0x7fff plus the lowest kept bit, then truncate.  A carry into the
   * exponent is the correct rounding (up to the next binade or to inf). */
  uint32_t lsb = (u >> 16) & 1u;
  u += 0x7fffu + lsb;
  return (uint16_t)(u >> 16);
}

static float load_elem(const void* base, size_t i, int dtype) {
  if (dtype == ORA_F32) return ((const float*)base)[i];
  return ora_bf16_to_f32(((const uint16_t*)base)[i]);
}

static void store_elem(void* base, size_t i, int dtype, float v) {
  if (dtype == ORA_F32)
    ((float*)base)[i] = v;
  else
    ((uint16_t*)base)[i] = ora_f32_to_bf16(v);
}

static size_t elem_size(int dtype) { return dtype == ORA_F32 ? 4 : 2; }

static int dtype_ok(int dtype) { return dtype == ORA_F32 || dtype == ORA_BF16; }

/* ---------------------------------------------------------------- gate -- */

int ora_topk_gate(const float* logits, int s, int e, int k, int renorm,
                  int32_t* idx, float* gate) {
  if (!logits || !idx || !gate || s < 0 || e < 1 || k < 1 || k > e) return ORA_EARG;
  for (size_t i = 0; i < (size_t)s * (size_t)e; ++i)
    if (!isfinite(logits[i])) return ORA_ENONFINITE;

#pragma omp parallel for schedule(static) num_threads(g_threads)
  for (int t = 0; t < s; ++t) {
    const float* l = logits + (size_t)t * e;
    int32_t* it = idx + (size_t)t * k;
    float* gt = gate + (size_t)t * k;
    /* position of each expert in the descending order, ties to the lower
     * index; the k experts with position < k are selected, in that order */
    for (int j = 0; j < e; ++j) {
      int pos = 0;
      for (int i = 0; i < e; ++i)
        if (l[i] > l[j] || (l[i] == l[j] && i < j)) ++pos;
      if (pos < k) it[pos] = j;
    }
    double M = (double)l[it[0]]; /* position 0 holds the largest logit */
    double den = 0.0;
    if (renorm) {
      for (int j = 0; j < k; ++j) den += exp((double)l[it[j]] - M);
    } else {
      for (int i = 0; i < e; ++i) den += exp((double)l[i] - M);
    }
    for (int j = 0; j < k; ++j) gt[j] = (float)(exp((double)l[it[j]] - M) / den);
  }
  return ORA_OK;
}

int ora_topk_gate_bwd(const float* logits, const int32_t* idx, const float* gate,
                      const float* dgate, int s, int e, int k, int renorm, float* dlogits) {
  if (!idx || !gate || !dgate || !dlogits || s < 0 || e < 1 || k < 1 || k > e) return ORA_EARG;
  if (!renorm && !logits) return ORA_EARG;
  if (!renorm)
    for (size_t i = 0; i < (size_t)s * (size_t)e; ++i)
      if (!isfinite(logits[i])) return ORA_ENONFINITE;
  for (size_t q = 0; q < (size_t)s * k; ++q)
    if (idx[q] < 0 || idx[q] >= e) return ORA_EROUTE;

#pragma omp parallel for schedule(static) num_threads(g_threads)
  for (int t = 0; t < s; ++t) {
    const int32_t* it = idx + (size_t)t * k;
    const float* gt = gate + (size_t)t * k;
    const float* dt = dgate + (size_t)t * k;
    float* out = dlogits + (size_t)t * e;
    double c = 0.0; /* sum_j g_j dgate_j */
    for (int j = 0; j < k; ++j) c += (double)gt[j] * (double)dt[j];
    if (renorm) {
      for (int i = 0; i < e; ++i) out[i] = 0.0f;
      for (int j = 0; j < k; ++j) out[it[j]] = (float)((double)gt[j] * ((double)dt[j] - c));
    } else {
      const float* l = logits + (size_t)t * e;
      double M = (double)l[0];
      for (int i = 1; i < e; ++i)
        if ((double)l[i] > M) M = (double)l[i];
      double den = 0.0;
      for (int i = 0; i < e; ++i) den += exp((double)l[i] - M);
      for (int i = 0; i < e; ++i) {
        double dg = 0.0;
        for (int j = 0; j < k; ++j)
          if (it[j] == i) dg = (double)dt[j];
        const double p = exp((double)l[i] - M) / den;
        out[i] = (float)(p * (dg - c));
      }
    }
  }
  return ORA_OK;
}

/* -------------------------------------------------------------- layout -- */

int ora_layout_ex(const int32_t* idx, int s, int e, int k, int capacity, int R, int priority,
                  int pad_multiple, int32_t* loc, int32_t* row, uint8_t* drop,
                  int32_t* raw_counts, int32_t* counts, int32_t* offsets,
                  uint8_t* token_in_rank, int32_t* rank_counts) {
  if (!idx || !loc || !row || !drop || !raw_counts || !counts || !offsets) return ORA_EARG;
  if (s < 0 || e < 1 || k < 1 || k > e || capacity < 0 || R < 0) return ORA_EARG;
  if (R > 0 && (e % R != 0 || !token_in_rank || !rank_counts)) return ORA_EARG;
  if ((priority != 0 && priority != 1) || pad_multiple < 1) return ORA_EARG;
  if (pad_multiple > 1 && capacity > 0) return ORA_EARG;

  /* every expert id in range and distinct within its token */
  for (int t = 0; t < s; ++t)
    for (int j = 0; j < k; ++j) {
      int32_t x = idx[(size_t)t * k + j];
      if (x < 0 || x >= e) return ORA_EROUTE;
      for (int jj = 0; jj < j; ++jj)
        if (idx[(size_t)t * k + jj] == x) return ORA_EROUTE;
    }

  /* location = running count of earlier routes to the same expert, in the
   * priority order: tokens in order (each token's routes together), or
   * route slot by route slot (all first choices, then all second ...) */
  int32_t* run = (int32_t*)calloc((size_t)e, sizeof(int32_t));
  if (!run) return ORA_EARG;
  if (priority == 0) {
    for (int t = 0; t < s; ++t)
      for (int j = 0; j < k; ++j) {
        int32_t x = idx[(size_t)t * k + j];
        loc[(size_t)t * k + j] = run[x];
        run[x] += 1;
      }
  } else {
    for (int j = 0; j < k; ++j)
      for (int t = 0; t < s; ++t) {
        int32_t x = idx[(size_t)t * k + j];
        loc[(size_t)t * k + j] = run[x];
        run[x] += 1;
      }
  }
  for (int x = 0; x < e; ++x) raw_counts[x] = run[x];
  free(run);

  if (capacity > 0) {
    for (int x = 0; x < e; ++x) counts[x] = raw_counts[x] < capacity ? raw_counts[x] : capacity;
    for (int x = 0; x <= e; ++x) offsets[x] = x * capacity;
    for (size_t r = 0; r < (size_t)s * k; ++r) {
      int dropped = loc[r] >= capacity;
      drop[r] = (uint8_t)dropped;
      row[r] = dropped ? -1 : idx[r] * capacity + loc[r];
    }
  } else {
    for (int x = 0; x < e; ++x) counts[x] = raw_counts[x];
    offsets[0] = 0;
    for (int x = 0; x < e; ++x) {
      int padded = (counts[x] + pad_multiple - 1) / pad_multiple * pad_multiple;
      offsets[x + 1] = offsets[x] + padded;
    }
    for (size_t r = 0; r < (size_t)s * k; ++r) {
      drop[r] = 0;
      row[r] = offsets[idx[r]] + loc[r];
    }
  }

  if (R > 0) {
    int per_rank = e / R;
    memset(token_in_rank, 0, (size_t)s * R);
    for (int r = 0; r < R; ++r) rank_counts[r] = 0;
    for (int t = 0; t < s; ++t) {
      for (int j = 0; j < k; ++j) {
        size_t q = (size_t)t * k + j;
        if (!drop[q]) token_in_rank[(size_t)t * R + idx[q] / per_rank] = 1;
      }
      for (int r = 0; r < R; ++r) rank_counts[r] += token_in_rank[(size_t)t * R + r];
    }
  }
  return ORA_OK;
}

int ora_layout(const int32_t* idx, int s, int e, int k, int capacity, int R,
               int32_t* loc, int32_t* row, uint8_t* drop,
               int32_t* raw_counts, int32_t* counts, int32_t* offsets,
               uint8_t* token_in_rank, int32_t* rank_counts) {
  return ora_layout_ex(idx, s, e, k, capacity, R, 0, 1, loc, row, drop, raw_counts, counts,
                       offsets, token_in_rank, rank_counts);
}

/* ---------------------------------------------------------- send slots -- */

int ora_rank_slots(const uint8_t* token_in_rank, int s, int R, int32_t* rank_slot) {
  if (!token_in_rank || !rank_slot || s < 0 || R < 1) return ORA_EARG;
  for (int r = 0; r < R; ++r) {
    int32_t next = 0; /* tokens seen so far that send to r */
    for (int t = 0; t < s; ++t) {
      if (token_in_rank[(size_t)t * R + r]) {
        rank_slot[(size_t)t * R + r] = next;
        next += 1;
      } else {
        rank_slot[(size_t)t * R + r] = -1;
      }
    }
  }
  return ORA_OK;
}

/* ------------------------------------------------------------ dispatch -- */

int ora_dispatch(const int32_t* row, int s, int k, int m, int dtype,
                 const void* x, int rows, void* X) {
  if (!row || !x || !X || s < 0 || k < 1 || m < 1 || rows < 0 || !dtype_ok(dtype)) return ORA_EARG;
  size_t es = elem_size(dtype);
  memset(X, 0, (size_t)rows * (size_t)m * es);
  for (size_t q = 0; q < (size_t)s * k; ++q)
    if (row[q] >= rows) return ORA_EARG;
#pragma omp parallel for schedule(static) num_threads(g_threads)
  for (int t = 0; t < s; ++t)
    for (int j = 0; j < k; ++j) {
      int32_t r = row[(size_t)t * k + j];
      if (r < 0) continue;
      memcpy((char*)X + (size_t)r * m * es, (const char*)x + (size_t)t * m * es, (size_t)m * es);
    }
  return ORA_OK;
}

/* ------------------------------------------------------------- combine -- */

int ora_combine(const int32_t* row, const float* gate, int s, int k, int m,
                int dtype, const void* y, void* out) {
  if (!row || !y || !out || s < 0 || k < 1 || m < 1 || !dtype_ok(dtype)) return ORA_EARG;
#pragma omp parallel for schedule(static) num_threads(g_threads)
  for (int t = 0; t < s; ++t)
    for (int c = 0; c < m; ++c) {
      float acc = 0.0f;
      for (int j = 0; j < k; ++j) {
        int32_t r = row[(size_t)t * k + j];
        if (r < 0) continue;
        float g = gate ? gate[(size_t)t * k + j] : 1.0f;
        acc = fmaf(g, load_elem(y, (size_t)r * m + c, dtype), acc);
      }
      store_elem(out, (size_t)t * m + c, dtype, acc);
    }
  return ORA_OK;
}

int ora_dispatch_bwd(const int32_t* row, int s, int k, int m, int dtype,
                     const void* dX, void* dx) {
  return ora_combine(row, NULL, s, k, m, dtype, dX, dx);
}

int ora_combine_bwd(const int32_t* row, const float* gate, int s, int k, int m,
                    int dtype, const void* dout, const void* y, int rows,
                    void* dY, float* dgate) {
  if (!row || !gate || !dout || !y || !dY || !dgate) return ORA_EARG;
  if (s < 0 || k < 1 || m < 1 || rows < 0 || !dtype_ok(dtype)) return ORA_EARG;
  size_t es = elem_size(dtype);
  memset(dY, 0, (size_t)rows * (size_t)m * es);
  for (size_t q = 0; q < (size_t)s * k; ++q)
    if (row[q] >= rows) return ORA_EARG;
#pragma omp parallel for schedule(static) num_threads(g_threads)
  for (int t = 0; t < s; ++t)
    for (int j = 0; j < k; ++j) {
      size_t q = (size_t)t * k + j;
      int32_t r = row[q];
      if (r < 0) {
        dgate[q] = 0.0f;
        continue;
      }
      double dot = 0.0;
      for (int c = 0; c < m; ++c) {
        float d = load_elem(dout, (size_t)t * m + c, dtype);
        float p = gate[q] * d; /* one fp32 multiply */
        store_elem(dY, (size_t)r * m + c, dtype, p);
        dot += (double)d * (double)load_elem(y, (size_t)r * m + c, dtype);
      }
      dgate[q] = (float)dot;
    }
  return ORA_OK;
}
