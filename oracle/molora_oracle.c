/*
 * molora_oracle.c -- plain, slow CPU definition of per-token adapter routing and the
 * batched LoRA apply.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the product path may call, link or execute this
 * file: only the test suite, the package smoke check and the benchmark's CPU-baseline /
 * reference arm use it.  It shares no code, header, table or helper with the CUDA path.
 *
 * Source: "MoLoRA: Composable Specialization via Per-Token Adapter Routing" (Shah & Wagle),
 * as printed on its paper pages (abstract, figure captions and tables).  Citations below
 * name the table or figure.
 *
 * Arithmetic: every sum is accumulated in double, in the order the definition states, and
 * rounded once at the end (to fp32 where the interface stores fp32).  bf16 inputs are
 * decoded exactly (a bf16 is the high half of an IEEE fp32).  No blocking, no reordering,
 * no fusion.  Compile with -ffp-contract=off so x86 and Arm hosts give identical bits.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define ORACLE_F32 0
#define ORACLE_BF16 1
#define ROUTER_HIDDEN 64 /* hidden width of the learned router: cost O(64d + 64K), Table 1 */

static double bf16_bits_to_double(uint16_t b) {
  uint32_t u = ((uint32_t)b) << 16;
  float f;
  memcpy(&f, &u, sizeof f);
  return (double)f;
}

/* Element i of a flat array of dtype f32 or bf16, exactly, as a double. */
static double elem(const void* p, int dtype, int64_t i) {
  if (dtype == ORACLE_BF16) return bf16_bits_to_double(((const uint16_t*)p)[i]);
  return (double)((const float*)p)[i];
}

/*
 * Vocabulary routing R_vocab(v) (Table 1, "Routing decision"; Table 12, disjoint vocabulary
 * ranges).  Adapter a owns the half-open range [starts[a], starts[a+1]).  A token outside
 * every range gets -1.  Plain linear scan over the ranges.
 * Returns the number of tokens that fell outside every range.
 */
int64_t oracle_route_vocab(const int32_t* tok, int64_t N, const int32_t* starts, int32_t K,
                           int32_t* adapter) {
  int64_t outside = 0;
  for (int64_t t = 0; t < N; ++t) {
    int32_t found = -1;
    for (int32_t a = 0; a < K; ++a) {
      if (starts[a] <= tok[t] && tok[t] < starts[a + 1]) {
        found = a;
        break;
      }
    }
    adapter[t] = found;
    if (found < 0) ++outside;
  }
  return outside;
}

/*
 * Learned router TopK(g(x)) (Table 1; Figure 2 left: the top-k adapters per token are
 * combined by a weighted sum; Table 10: softmax(Wx + b) gating).
 *   hidden_j = max(0, sum_i x_i W1[i,j] + b1_j)          j < 64, kept in double
 *   logit_a  = fp32( sum_j hidden_j W2[j,a] + b2_a )     a < K
 *   selection: indices ordered by (logit descending, index ascending), first k kept
 *   weight_j = exp(l_j - l_max) / sum over the k selected of exp(l - l_max), rounded to fp32
 * x, W1 and W2 share `dtype`; b1 and b2 are fp32 or NULL (zero).  `logits` may be NULL.
 * ids and w are [N x k] row-major, in selection order.
 */
void oracle_router_topk(const void* x, int dtype, int64_t N, int32_t d_in, const void* W1,
                        const float* b1, const void* W2, const float* b2, int32_t K, int32_t k,
                        float* logits, int32_t* ids, float* w) {
  double hidden[ROUTER_HIDDEN];
  float* lg = (float*)malloc(sizeof(float) * (size_t)K);
  int32_t* order = (int32_t*)malloc(sizeof(int32_t) * (size_t)K);
  for (int64_t t = 0; t < N; ++t) {
    for (int j = 0; j < ROUTER_HIDDEN; ++j) {
      double s = 0.0;
      for (int32_t i = 0; i < d_in; ++i)
        s += elem(x, dtype, t * (int64_t)d_in + i) * elem(W1, dtype, (int64_t)i * ROUTER_HIDDEN + j);
      if (b1) s += (double)b1[j];
      hidden[j] = s > 0.0 ? s : 0.0;
    }
    for (int32_t a = 0; a < K; ++a) {
      double s = 0.0;
      for (int j = 0; j < ROUTER_HIDDEN; ++j) s += hidden[j] * elem(W2, dtype, (int64_t)j * K + a);
      if (b2) s += (double)b2[a];
      lg[a] = (float)s;
      if (logits) logits[t * K + a] = lg[a];
    }
    /* stable insertion sort of indices by descending fp32 logit: equal logits keep
       ascending index order */
    for (int32_t a = 0; a < K; ++a) {
      int32_t p = a;
      while (p > 0 && lg[order[p - 1]] < lg[a]) {
        order[p] = order[p - 1];
        --p;
      }
      order[p] = a;
    }
    double lmax = (double)lg[order[0]];
    double denom = 0.0;
    for (int32_t j = 0; j < k; ++j) denom += exp((double)lg[order[j]] - lmax);
    for (int32_t j = 0; j < k; ++j) {
      ids[t * k + j] = order[j];
      w[t * k + j] = (float)(exp((double)lg[order[j]] - lmax) / denom);
    }
  }
  free(lg);
  free(order);
}

/*
 * Dispatch (Table 1: histogram computation, pointer arrays; Figure 2 right: tokens are
 * grouped by their selected adapter).  Slot s = t*k + j is token t's j-th choice.
 *   counts[a]    = number of slots with ids[s] == a
 *   offsets[0]   = 0, offsets[a+1] = offsets[a] + counts[a]
 *   perm[offsets[a] + q] = the q-th slot (in ascending s) whose id is a   (stable)
 * Slots with an id outside [0, K) are left out; perm entries past offsets[K] are -1.
 * Returns the number of slots left out.
 */
int64_t oracle_dispatch(const int32_t* ids, int64_t N, int32_t k, int32_t K, int32_t* counts,
                        int32_t* offsets, int32_t* perm) {
  int64_t S = N * (int64_t)k;
  int64_t invalid = 0;
  for (int32_t a = 0; a < K; ++a) counts[a] = 0;
  for (int64_t s = 0; s < S; ++s) {
    if (ids[s] >= 0 && ids[s] < K)
      counts[ids[s]] += 1;
    else
      ++invalid;
  }
  offsets[0] = 0;
  for (int32_t a = 0; a < K; ++a) offsets[a + 1] = offsets[a] + counts[a];
  int32_t* fill = (int32_t*)malloc(sizeof(int32_t) * (size_t)K);
  for (int32_t a = 0; a < K; ++a) fill[a] = offsets[a];
  for (int64_t s = 0; s < S; ++s) perm[s] = -1;
  for (int64_t s = 0; s < S; ++s) {
    int32_t a = ids[s];
    if (a >= 0 && a < K) perm[fill[a]++] = (int32_t)s;
  }
  free(fill);
  return invalid;
}

/*
 * Per-token LoRA apply, the plain token-major definition (Figure 2 left; Table 10 weight
 * shapes A: (K, d_in, r), B: (K, r, d_out)):
 *   y[t,:] = fp32( y0[t,:] + sum_j scale * w[t,j] * (x[t,:] A_{ids[t,j]}) B_{ids[t,j]} )
 * One double accumulator per output element, one rounding.  w == NULL means every weight
 * is 1.  Slots whose id is outside [0, K) add nothing.  `work` (may be NULL) receives the
 * number of adapter-rows evaluated: one per valid slot, i.e. N*k, never K*N.
 */
void oracle_lora_apply(const void* x, int dtype, int64_t N, int32_t d_in, int32_t d_out,
                       const void* A, const void* B, int32_t K, int32_t r, const int32_t* ids,
                       const float* w, int32_t k, float scale, float* y, int64_t* work) {
  double* acc = (double*)malloc(sizeof(double) * (size_t)d_out);
  double* h = (double*)malloc(sizeof(double) * (size_t)r);
  int64_t rows = 0;
  for (int64_t t = 0; t < N; ++t) {
    for (int32_t o = 0; o < d_out; ++o) acc[o] = (double)y[t * d_out + o];
    for (int32_t j = 0; j < k; ++j) {
      int32_t a = ids[t * k + j];
      if (a < 0 || a >= K) continue;
      ++rows;
      double coef = (double)scale * (w ? (double)w[t * k + j] : 1.0);
      for (int32_t q = 0; q < r; ++q) {
        double s = 0.0;
        for (int32_t i = 0; i < d_in; ++i)
          s += elem(x, dtype, t * (int64_t)d_in + i) *
               elem(A, dtype, ((int64_t)a * d_in + i) * r + q);
        h[q] = s;
      }
      for (int32_t o = 0; o < d_out; ++o) {
        double s = 0.0;
        for (int32_t q = 0; q < r; ++q) s += h[q] * elem(B, dtype, ((int64_t)a * r + q) * d_out + o);
        acc[o] += coef * s;
      }
    }
    for (int32_t o = 0; o < d_out; ++o) y[t * d_out + o] = (float)acc[o];
  }
  if (work) *work += rows;
  free(acc);
  free(h);
}

/*
 * One masked per-sequence pass (Table 3 / Table 7: per-sequence routing needs K passes for
 * a K-modality workload): adapter `a` is evaluated for EVERY token and the result is
 * multiplied by the mask [adapter_of[t] == a] before it is added:
 *   y[t,:] = fp32( y[t,:] + mask_t * scale * (x[t,:] A_a) B_a )
 * `work` (may be NULL) receives N adapter-rows: the whole batch, masked or not.
 */
void oracle_masked_pass(const void* x, int dtype, int64_t N, int32_t d_in, int32_t d_out,
                        const void* A, const void* B, int32_t K, int32_t r,
                        const int32_t* adapter_of, int32_t a, float scale, float* y,
                        int64_t* work) {
  (void)K;
  double* h = (double*)malloc(sizeof(double) * (size_t)r);
  for (int64_t t = 0; t < N; ++t) {
    double mask = adapter_of[t] == a ? 1.0 : 0.0;
    for (int32_t q = 0; q < r; ++q) {
      double s = 0.0;
      for (int32_t i = 0; i < d_in; ++i)
        s += elem(x, dtype, t * (int64_t)d_in + i) * elem(A, dtype, ((int64_t)a * d_in + i) * r + q);
      h[q] = s;
    }
    for (int32_t o = 0; o < d_out; ++o) {
      double s = 0.0;
      for (int32_t q = 0; q < r; ++q) s += h[q] * elem(B, dtype, ((int64_t)a * r + q) * d_out + o);
      y[t * d_out + o] = (float)((double)y[t * d_out + o] + mask * (double)scale * s);
    }
  }
  if (work) *work += N;
  free(h);
}
