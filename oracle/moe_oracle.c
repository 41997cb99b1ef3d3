/*
 * CPU oracle for the routed-expert MoE FFN layer with sigmoid routing.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing on the product path links, loads or
 * calls this file: only the tests, the smoke check and the benchmark's CPU
 * baseline leg do.  It shares no code with the CUDA library.
 *
 * What the layer computes, as the GLM-5.3-Flash pages describe it:
 *   - "Add GLM-5.3-Flash (glm5next) support with ROCmFP mix qtypes (105/106)"
 *     (lucebox PR #1), section "MoE FFN (REAL routed expert execution)":
 *     sigmoid routing over the router logits plus a per-expert bias, top-8
 *     selection, weight normalisation, per-expert gate / up / down matmuls, a
 *     clamped SwiGLU between gate/up and down, and a shared expert combined
 *     with the routed output.
 *   - same page, section "Architecture": 288 routed experts, top-8, one shared
 *     expert; clamped SwiGLU with the gate limited to (-inf, 10] before the
 *     SiLU and the up projection to [-10, 10].
 *   - same page, section "What Executes vs. TODO", item 3 "MoE expert
 *     evaluation": the weighted combination of expert outputs and the shared
 *     expert.
 *   - "feat(glm53): add device-resident HIP backend for MI350P" (colibri
 *     PR #1448), section "Key changes": deterministic top-k routing, and the
 *     grouped fmt=4 Int4 weights decoded as offset-binary (nibble - 8).
 *
 * Precision.  The router logits are accumulated in float (h ascending), the
 * precision the GPU path accumulates in, so that both sides take the top-8
 * decision on float logits.  Everything after that (sigmoid, normalisation,
 * expert matmuls, SwiGLU, combination) is computed in double.  bf16 values
 * and Int4 codes are widened element by element; no blocking or reordering
 * beyond the sums written below.
 *
 * Readings where the pages are silent (each also listed in the design notes):
 *   - the bias sits inside the sigmoid and the biased score is used both to
 *     select and to weight (the page writes sigmoid(moe_gate @ input +
 *     moe_exp_probs_b) and nothing else);
 *   - "weight normalization" divides the 8 selected scores by their sum; no
 *     epsilon and no extra routed scaling factor;
 *   - ties in the top-8 go to the lower expert index; slots are emitted in
 *     descending score order;
 *   - the shared expert uses the same clamped SwiGLU and enters with weight 1;
 *   - Int4 grouping: 32 consecutive reduction-dimension elements share one
 *     bf16 scale; element 2m of a row sits in the low nibble of byte m.
 *
 * Storage conventions (all row-major):
 *   x      [T][H]   bf16 bits       router weight [E][H] bf16 bits
 *   bias   [E]      float
 *   gate, up  [E][I][H]  (output-major "nn.Linear" layout, H contiguous)
 *   down      [E][H][I]
 *   Int4: codes [E][N][K/2] uint8, scales [E][N][K/32] bf16 bits, where
 *   N x K is the matrix shape above.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

#define ORACLE_FMT_BF16 0
#define ORACLE_FMT_INT4_G32 1
#define ORACLE_INT4_GROUP 32

/* ------------------------------------------------------------ widening */

double oracle_bf16_to_double(uint16_t bits) {
  uint32_t u = (uint32_t)bits << 16;
  float f;
  memcpy(&f, &u, sizeof f);
  return (double)f;
}

/* Offset-binary Int4 ("nibble - 8", colibri PR #1448, Key changes). */
int oracle_int4_decode(int nibble) { return (nibble & 15) - 8; }

/* Element (n, k) of one N x K matrix in the chosen storage. */
static double weight_at(int fmt, const void* w, const uint16_t* scale, int64_t K,
                        int64_t n, int64_t k) {
  if (fmt == ORACLE_FMT_BF16) return oracle_bf16_to_double(((const uint16_t*)w)[n * K + k]);
  const uint8_t byte = ((const uint8_t*)w)[n * (K / 2) + k / 2];
  const int nibble = (k & 1) ? (byte >> 4) : (byte & 15);
  const double s = oracle_bf16_to_double(scale[n * (K / ORACLE_INT4_GROUP) + k / ORACLE_INT4_GROUP]);
  return (double)oracle_int4_decode(nibble) * s;
}

double oracle_weight_element(int fmt, const void* w, const uint16_t* scale, int64_t K,
                             int64_t n, int64_t k) {
  return weight_at(fmt, w, scale, K, n, k);
}

/* ------------------------------------------------------------ router */

/* z[t][e] = (sum over h of x[t][h] * Wr[e][h], in float, h ascending) + b[e] */
void oracle_router_logits(int64_t T, int64_t H, int64_t E, const uint16_t* x,
                          const uint16_t* w_router, const float* b, float* z) {
#pragma omp parallel for schedule(static)
  for (int64_t t = 0; t < T; ++t)
    for (int64_t e = 0; e < E; ++e) {
      float acc = 0.0f;
      for (int64_t h = 0; h < H; ++h)
        acc += (float)oracle_bf16_to_double(x[t * H + h]) *
               (float)oracle_bf16_to_double(w_router[e * H + h]);
      z[t * E + e] = acc + b[e];
    }
}

double oracle_sigmoid(double z) { return 1.0 / (1.0 + exp(-z)); }

typedef struct {
  float z;
  int32_t e;
} scored;

/* higher score first; equal scores: lower expert index first */
static int by_score_then_index(const void* pa, const void* pb) {
  const scored* a = (const scored*)pa;
  const scored* b = (const scored*)pb;
  if (a->z > b->z) return -1;
  if (a->z < b->z) return 1;
  return (a->e > b->e) - (a->e < b->e);
}

/*
 * Top-k by a full sort of all E experts on (score desc, index asc).  The
 * sigmoid is strictly increasing, so ordering by the logit orders by the
 * routing probability.  Selected weights: s_j / sum_j' s_j', the sum taken in
 * slot order.  s_sel (optional) receives the unnormalised sigmoid scores.
 */
void oracle_topk(int64_t T, int64_t E, int64_t k, const float* z, int32_t* idx,
                 double* w, double* s_sel) {
#pragma omp parallel
  {
    scored* buf = (scored*)malloc(sizeof(scored) * (size_t)E);
#pragma omp for schedule(static)
    for (int64_t t = 0; t < T; ++t) {
      for (int64_t e = 0; e < E; ++e) {
        buf[e].z = z[t * E + e];
        buf[e].e = (int32_t)e;
      }
      qsort(buf, (size_t)E, sizeof(scored), by_score_then_index);
      double s[64];
      double sum = 0.0;
      for (int64_t j = 0; j < k; ++j) {
        s[j] = oracle_sigmoid((double)buf[j].z);
        sum += s[j];
      }
      for (int64_t j = 0; j < k; ++j) {
        idx[t * k + j] = buf[j].e;
        w[t * k + j] = s[j] / sum;
        if (s_sel) s_sel[t * k + j] = s[j];
      }
    }
    free(buf);
  }
}

/* ------------------------------------------------------------ permutation */

/*
 * Grouping of the (token, slot) pairs by expert, the shared expert appended
 * as group E holding every token.
 *   cnt[e]      = number of (t, j) with idx[t][j] == e;  cnt[E] = T
 *   offsets     = exclusive prefix sum of cnt, length E + 2 (last = (k+1)T)
 *   rows of a group are ordered by ascending token
 *   gather[r]   = token of row r
 *   row_of[t][j]= row holding (t, j)
 */
void oracle_permute(int64_t T, int64_t E, int64_t k, const int32_t* idx, int32_t* offsets,
                    int32_t* gather, int32_t* row_of) {
  int64_t* cnt = (int64_t*)calloc((size_t)(E + 1), sizeof(int64_t));
  for (int64_t t = 0; t < T; ++t)
    for (int64_t j = 0; j < k; ++j) cnt[idx[t * k + j]] += 1;
  cnt[E] = T;
  int64_t run = 0;
  for (int64_t e = 0; e <= E; ++e) {
    offsets[e] = (int32_t)run;
    run += cnt[e];
  }
  offsets[E + 1] = (int32_t)run;
  int64_t* fill = (int64_t*)calloc((size_t)(E + 1), sizeof(int64_t));
  for (int64_t t = 0; t < T; ++t) { /* ascending t keeps each group ordered */
    for (int64_t j = 0; j < k; ++j) {
      const int64_t e = idx[t * k + j];
      const int64_t r = offsets[e] + fill[e]++;
      gather[r] = (int32_t)t;
      row_of[t * k + j] = (int32_t)r;
    }
    gather[offsets[E] + t] = (int32_t)t;
  }
  free(cnt);
  free(fill);
}

/* ------------------------------------------------------------ expert FFN */

/* silu(min(g, 10)) * clamp(u, -10, 10), with silu(v) = v / (1 + exp(-v)) */
double oracle_clamped_swiglu(double g, double u) {
  const double gc = g < 10.0 ? g : 10.0;
  const double uc = u < -10.0 ? -10.0 : (u > 10.0 ? 10.0 : u);
  return gc / (1.0 + exp(-gc)) * uc;
}

/*
 * One expert applied to one token vector xv[H] (double):
 *   g_i = sum_h xv_h Wg[i][h],  u_i = sum_h xv_h Wu[i][h]
 *   a_i = clamped_swiglu(g_i, u_i)
 *   y_n = sum_i a_i Wd[n][i]
 * The matrix pointers address this expert's own [I][H], [I][H], [H][I] slabs
 * (or codes / scales of the same shapes).  act (optional) receives a[I].
 */
void oracle_expert_ffn(int64_t H, int64_t I, int fmt, const void* gate, const void* up,
                       const void* down, const uint16_t* gate_scale, const uint16_t* up_scale,
                       const uint16_t* down_scale, const double* xv, double* y, double* act) {
  double* a = (double*)malloc(sizeof(double) * (size_t)I);
  for (int64_t i = 0; i < I; ++i) {
    double g = 0.0, u = 0.0;
    for (int64_t h = 0; h < H; ++h) {
      g += xv[h] * weight_at(fmt, gate, gate_scale, H, i, h);
      u += xv[h] * weight_at(fmt, up, up_scale, H, i, h);
    }
    a[i] = oracle_clamped_swiglu(g, u);
    if (act) act[i] = a[i];
  }
  for (int64_t n = 0; n < H; ++n) {
    double acc = 0.0;
    for (int64_t i = 0; i < I; ++i) acc += a[i] * weight_at(fmt, down, down_scale, I, n, i);
    y[n] = acc;
  }
  free(a);
}

/* Byte offset of expert e's slab for an N x K matrix in the chosen storage. */
static size_t slab_bytes(int fmt, int64_t N, int64_t K) {
  return fmt == ORACLE_FMT_BF16 ? (size_t)(N * K) * 2 : (size_t)(N * K) / 2;
}
static size_t scale_elems(int64_t N, int64_t K) { return (size_t)(N * (K / ORACLE_INT4_GROUP)); }

typedef struct {
  const void *gate, *up, *down;
  const uint16_t *gate_scale, *up_scale, *down_scale;
} oracle_weights;

static void expert_ffn_of(int64_t H, int64_t I, int fmt, const oracle_weights* w, int64_t e,
                          const double* xv, double* y) {
  const size_t gb = slab_bytes(fmt, I, H), db = slab_bytes(fmt, H, I);
  const size_t gs = scale_elems(I, H), ds = scale_elems(H, I);
  const int q = fmt != ORACLE_FMT_BF16;
  oracle_expert_ffn(H, I, fmt, (const char*)w->gate + e * gb, (const char*)w->up + e * gb,
                    (const char*)w->down + e * db, q ? w->gate_scale + e * gs : NULL,
                    q ? w->up_scale + e * gs : NULL, q ? w->down_scale + e * ds : NULL, xv, y,
                    NULL);
}

/*
 * The whole layer for T tokens:
 *   out[t] = sum_j w[t][j] * FFN_{idx[t][j]}(x_t) + FFN_shared(x_t)
 * with the sum taken over j = 0..k-1 and the shared term added last.
 * Optional outputs: idx [T][k], w [T][k], y_perm [(k+1)T][H] (the unweighted
 * per-row expert outputs in the row order of oracle_permute).
 * nthreads <= 0 keeps the OpenMP default.
 */
int oracle_moe_forward(int64_t T, int64_t H, int64_t E, int64_t I, int64_t I_shared, int64_t k,
                       int fmt, const uint16_t* x, const uint16_t* w_router, const float* b,
                       const void* gate, const void* up, const void* down,
                       const uint16_t* gate_scale, const uint16_t* up_scale,
                       const uint16_t* down_scale, const void* s_gate, const void* s_up,
                       const void* s_down, const uint16_t* s_gate_scale,
                       const uint16_t* s_up_scale, const uint16_t* s_down_scale,
                       int32_t* idx_out, double* w_out, double* out, int nthreads) {
  if (k <= 0 || k > 64 || k > E || (fmt != ORACLE_FMT_BF16 && fmt != ORACLE_FMT_INT4_G32))
    return 1;
  if (fmt == ORACLE_FMT_INT4_G32 &&
      (H % ORACLE_INT4_GROUP || I % ORACLE_INT4_GROUP || I_shared % ORACLE_INT4_GROUP))
    return 1;
#ifdef _OPENMP
  if (nthreads > 0) omp_set_num_threads(nthreads);
#else
  (void)nthreads;
#endif
  const oracle_weights routed = {gate, up, down, gate_scale, up_scale, down_scale};
  const oracle_weights shared = {s_gate, s_up, s_down, s_gate_scale, s_up_scale, s_down_scale};

  float* z = (float*)malloc(sizeof(float) * (size_t)(T * E));
  int32_t* idx = idx_out ? idx_out : (int32_t*)malloc(sizeof(int32_t) * (size_t)(T * k));
  double* w = w_out ? w_out : (double*)malloc(sizeof(double) * (size_t)(T * k));
  oracle_router_logits(T, H, E, x, w_router, b, z);
  oracle_topk(T, E, k, z, idx, w, NULL);

#pragma omp parallel
  {
    double* xv = (double*)malloc(sizeof(double) * (size_t)H);
    double* y = (double*)malloc(sizeof(double) * (size_t)H);
#pragma omp for schedule(dynamic, 1)
    for (int64_t t = 0; t < T; ++t) {
      for (int64_t h = 0; h < H; ++h) xv[h] = oracle_bf16_to_double(x[t * H + h]);
      double* o = out + t * H;
      for (int64_t h = 0; h < H; ++h) o[h] = 0.0;
      for (int64_t j = 0; j < k; ++j) {
        expert_ffn_of(H, I, fmt, &routed, idx[t * k + j], xv, y);
        const double wj = w[t * k + j];
        for (int64_t h = 0; h < H; ++h) o[h] += wj * y[h];
      }
      expert_ffn_of(H, I_shared, fmt, &shared, 0, xv, y);
      for (int64_t h = 0; h < H; ++h) o[h] += y[h];
    }
    free(xv);
    free(y);
  }
  free(z);
  if (!idx_out) free(idx);
  if (!w_out) free(w);
  return 0;
}

/*
 * Unweighted per-row expert outputs in permuted row order (the quantity the
 * grouped expert stage produces before combination):
 *   y_perm[r] = FFN_{group(r)}(x_{gather[r]}),  group E = the shared expert.
 * offsets / gather come from oracle_permute.  Rows [r0, r1) only.
 */
void oracle_expert_rows(int64_t T, int64_t H, int64_t E, int64_t I, int64_t I_shared, int fmt,
                        const uint16_t* x, const int32_t* offsets, const int32_t* gather,
                        const void* gate, const void* up, const void* down,
                        const uint16_t* gate_scale, const uint16_t* up_scale,
                        const uint16_t* down_scale, const void* s_gate, const void* s_up,
                        const void* s_down, const uint16_t* s_gate_scale,
                        const uint16_t* s_up_scale, const uint16_t* s_down_scale, int64_t r0,
                        int64_t r1, double* y_rows) {
  (void)T;
  const oracle_weights routed = {gate, up, down, gate_scale, up_scale, down_scale};
  const oracle_weights shared = {s_gate, s_up, s_down, s_gate_scale, s_up_scale, s_down_scale};
#pragma omp parallel
  {
    double* xv = (double*)malloc(sizeof(double) * (size_t)H);
#pragma omp for schedule(dynamic, 1)
    for (int64_t r = r0; r < r1; ++r) {
      int64_t g = 0;
      while (g < E && offsets[g + 1] <= r) ++g; /* group holding row r */
      const int64_t t = gather[r];
      for (int64_t h = 0; h < H; ++h) xv[h] = oracle_bf16_to_double(x[t * H + h]);
      if (g < E)
        expert_ffn_of(H, I, fmt, &routed, g, xv, y_rows + (r - r0) * H);
      else
        expert_ffn_of(H, I_shared, fmt, &shared, 0, xv, y_rows + (r - r0) * H);
    }
    free(xv);
  }
}

/*
 * Combination of per-row outputs:
 *   out[t] = sum_j w[t][j] * y_perm[row_of[t][j]] + y_perm[shared_row0 + t]
 * j ascending, shared term last.
 */
void oracle_combine(int64_t T, int64_t H, int64_t k, const double* y_perm, const int32_t* row_of,
                    const double* w, int64_t shared_row0, double* out) {
  for (int64_t t = 0; t < T; ++t)
    for (int64_t h = 0; h < H; ++h) {
      double acc = 0.0;
      for (int64_t j = 0; j < k; ++j) acc += w[t * k + j] * y_perm[(int64_t)row_of[t * k + j] * H + h];
      out[t * H + h] = acc + y_perm[(shared_row0 + t) * H + h];
    }
}

int oracle_max_threads(void) {
#ifdef _OPENMP
  return omp_get_max_threads();
#else
  return 1;
#endif
}
