/*
 * CPU oracle for the forward pass of one Mixture-of-Experts FFN layer.
 *
 * TEST INFRASTRUCTURE ONLY.  This file is the plain, slow, obviously correct
 * definition the CUDA path is checked against.  It shares no code, header or
 * constant with the CUDA library; only the test suite, the smoke check and the
 * benchmark's CPU-baseline leg load it.
 *
 * Everything is evaluated in double precision over bf16-decoded (exact)
 * inputs, one step at a time, in the order the pages state the method:
 *
 *   router       s = W_r x                      ("MoE推理优化全景指南", section
 *                                                 "从 Dense FFN 到专家集合")
 *   top-k gating three variants                  (CS349D lecture 8, section 1.2
 *                                                 "MoE 层的结构")
 *   dispatch     histogram / prefix sum / permute ("MoE推理优化全景指南", section
 *                                                 "Dispatch 并不是一次普通 all-to-all")
 *   expert FFN   SwiGLU with W_gate/up[2I,H], W_down[H,I]
 *                                                (Moebius reading notes, eq. (2);
 *                                                 Moebius paper, "Weights Resharding")
 *   combine      y = sum_i g_i * FFN_i(x)        (Moebius reading notes, eq. (1))
 *
 * Readings where the pages leave a step open (each is listed with its reason
 * in the design notes):
 *   - router logits are float32: the exact double dot product rounded once;
 *     the expert selection is decided on those float32 values;
 *   - ties in the selection go to the lower expert index; slot order within a
 *     token is the selection order (best first);
 *   - the sigmoid variant selects on float32(float32(sigmoid(s)) + b) and
 *     weights with sigmoid(s) only (the bias changes who is chosen, not how
 *     much);
 *   - W13 rows [0,I) are the gate projection, rows [I,2I) the up projection,
 *     h = SiLU(gate) * up, SiLU(z) = z / (1 + e^-z);
 *   - inside one expert's segment, assignments keep ascending token order;
 *   - the shared expert (if any) is added with weight 1.
 *
 * Parity pins (tests/test_oracle_pins.py) tie each function to something other
 * than itself: the pages' worked examples, closed forms, invariants and the
 * dense-FFN special case.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

enum { GATE_TOPK_SOFTMAX = 0, GATE_SOFTMAX_TOPK = 1, GATE_SOFTMAX_TOPK_RENORM = 2,
       GATE_SIGMOID_BIAS_RENORM = 3 };

/* bf16 is the upper half of an IEEE float32: widen and convert (exact). */
static double bf16_value(uint16_t v) {
    uint32_t u = (uint32_t)v << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

static double sigmoid(double z) { return 1.0 / (1.0 + exp(-z)); }

int oracle_max_threads(void) {
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

/* Router: s[t,e] = float32( sum_h W_r[e,h] * x[t,h] ), the sum in double. */
void oracle_router_logits(const uint16_t *x, const float *w_router, int64_t T, int64_t H,
                          int64_t E, float *s_out, int nthreads) {
#ifdef _OPENMP
#pragma omp parallel for num_threads(nthreads > 0 ? nthreads : 1) schedule(static)
#endif
    for (int64_t t = 0; t < T; ++t) {
        for (int64_t e = 0; e < E; ++e) {
            double acc = 0.0;
            for (int64_t h = 0; h < H; ++h)
                acc += (double)w_router[e * H + h] * bf16_value(x[t * H + h]);
            s_out[t * E + e] = (float)acc;
        }
    }
    (void)nthreads;
}

typedef struct { float key; int32_t idx; } ranked_t;

/* best first: larger key first, equal keys -> lower index first */
static int rank_cmp(const void *pa, const void *pb) {
    const ranked_t *a = (const ranked_t *)pa, *b = (const ranked_t *)pb;
    if (a->key > b->key) return -1;
    if (a->key < b->key) return 1;
    return (a->idx < b->idx) ? -1 : (a->idx > b->idx);
}

/*
 * Top-k selection and gate weights for each token.
 *   ids[t,j]  j-th selected expert (best first)
 *   w[t,j]    its gate weight (double)
 *   gap[t]    selection key of the k-th minus that of the (k+1)-th expert;
 *             NAN when k == E (no boundary)
 * Returns 0, or -1 on bad arguments.
 */
int oracle_topk_gating(const float *s, const float *sel_bias, int64_t T, int64_t E, int64_t k,
                       int mode, int32_t *ids, double *w, double *gap) {
    if (k < 1 || k > E || mode < 0 || mode > 3) return -1;
    if (mode == GATE_SIGMOID_BIAS_RENORM && sel_bias == NULL) return -1;
    ranked_t *r = (ranked_t *)malloc((size_t)E * sizeof(ranked_t));
    double *p = (double *)malloc((size_t)E * sizeof(double));
    if (!r || !p) { free(r); free(p); return -1; }
    for (int64_t t = 0; t < T; ++t) {
        const float *st = s + t * E;
        /* selection key */
        for (int64_t e = 0; e < E; ++e) {
            float key = st[e];
            if (mode == GATE_SIGMOID_BIAS_RENORM) {
                float a = (float)sigmoid((double)st[e]);
                key = (float)(a + sel_bias[e]);   /* float32 add, rounded once */
            }
            r[e].key = key;
            r[e].idx = (int32_t)e;
        }
        qsort(r, (size_t)E, sizeof(ranked_t), rank_cmp);
        for (int64_t j = 0; j < k; ++j) ids[t * k + j] = r[j].idx;
        gap[t] = (k < E) ? (double)r[k - 1].key - (double)r[k].key : NAN;

        /* gate weights */
        if (mode == GATE_TOPK_SOFTMAX) {
            /* softmax over the kept logits only (the others are -inf) */
            double m = -INFINITY, z = 0.0;
            for (int64_t j = 0; j < k; ++j) m = fmax(m, (double)st[r[j].idx]);
            for (int64_t j = 0; j < k; ++j) z += exp((double)st[r[j].idx] - m);
            for (int64_t j = 0; j < k; ++j) w[t * k + j] = exp((double)st[r[j].idx] - m) / z;
        } else if (mode == GATE_SOFTMAX_TOPK || mode == GATE_SOFTMAX_TOPK_RENORM) {
            /* softmax over all E experts, then keep the selected probabilities */
            double m = -INFINITY, z = 0.0;
            for (int64_t e = 0; e < E; ++e) m = fmax(m, (double)st[e]);
            for (int64_t e = 0; e < E; ++e) { p[e] = exp((double)st[e] - m); z += p[e]; }
            for (int64_t e = 0; e < E; ++e) p[e] /= z;
            double kept = 0.0;
            for (int64_t j = 0; j < k; ++j) kept += p[r[j].idx];
            for (int64_t j = 0; j < k; ++j)
                w[t * k + j] = (mode == GATE_SOFTMAX_TOPK) ? p[r[j].idx] : p[r[j].idx] / kept;
        } else {
            /* sigmoid affinities of the selected experts, renormalised; no bias */
            double kept = 0.0;
            for (int64_t j = 0; j < k; ++j) kept += sigmoid((double)st[r[j].idx]);
            for (int64_t j = 0; j < k; ++j) w[t * k + j] = sigmoid((double)st[r[j].idx]) / kept;
        }
    }
    free(r);
    free(p);
    return 0;
}

/*
 * Dispatch layout from the flat assignment list a = t*k + j -> expert ids[a].
 *   counts[e]        number of assignments to expert e         (histogram)
 *   offsets[e]       sum of counts of experts < e; offsets[E] = T*k  (prefix sum)
 *   perm_src[p]      the assignment stored at position p: positions
 *                    [offsets[e], offsets[e+1]) hold expert e's assignments in
 *                    ascending token order                       (permute)
 *   inv_pos[a]       the position of assignment a                (inverse)
 * Returns 0, or -1 if an id is out of range.
 */
int oracle_dispatch(const int32_t *ids, int64_t T, int64_t k, int64_t E, int32_t *counts,
                    int32_t *offsets, int32_t *perm_src, int32_t *inv_pos) {
    const int64_t Na = T * k;
    for (int64_t a = 0; a < Na; ++a)
        if (ids[a] < 0 || ids[a] >= E) return -1;
    for (int64_t e = 0; e < E; ++e) counts[e] = 0;
    for (int64_t a = 0; a < Na; ++a) counts[ids[a]] += 1;
    offsets[0] = 0;
    for (int64_t e = 0; e < E; ++e) offsets[e + 1] = offsets[e] + counts[e];
    int64_t p = 0;
    for (int64_t e = 0; e < E; ++e)
        for (int64_t a = 0; a < Na; ++a)
            if (ids[a] == e) { perm_src[p] = (int32_t)a; inv_pos[a] = (int32_t)p; ++p; }
    return 0;
}

/* Imbalance ratio max_e n_e / (N_a / E) as the exact fraction num/den. */
void oracle_imbalance(const int32_t *counts, int64_t E, int64_t Na, int64_t *num, int64_t *den) {
    int64_t mx = 0;
    for (int64_t e = 0; e < E; ++e) if (counts[e] > mx) mx = counts[e];
    int64_t a = mx * E, b = Na;
    int64_t g0 = a, g1 = b;
    while (g1 != 0) { int64_t t = g0 % g1; g0 = g1; g1 = t; }
    if (g0 == 0) g0 = 1;
    *num = a / g0;
    *den = b / g0;
}

/*
 * One expert's SwiGLU FFN on one token, in double:
 *   g = W13[0:I] x,  u = W13[I:2I] x,  h = SiLU(g) * u,  out = W2 h
 * w13: [2I,H] bf16, w2: [H,I] bf16, x: [H] bf16, out: [H] double.
 */
void oracle_expert_ffn(const uint16_t *x, const uint16_t *w13, const uint16_t *w2, int64_t H,
                       int64_t I, double *out) {
    double *h = (double *)malloc((size_t)I * sizeof(double));
    for (int64_t i = 0; i < I; ++i) {
        double g = 0.0, u = 0.0;
        for (int64_t c = 0; c < H; ++c) {
            double xv = bf16_value(x[c]);
            g += bf16_value(w13[i * H + c]) * xv;
            u += bf16_value(w13[(I + i) * H + c]) * xv;
        }
        h[i] = g * sigmoid(g) * u;
    }
    for (int64_t r = 0; r < H; ++r) {
        double acc = 0.0;
        for (int64_t i = 0; i < I; ++i) acc += bf16_value(w2[r * I + i]) * h[i];
        out[r] = acc;
    }
    free(h);
}

/*
 * Layer output for a list of tokens:
 *   y[n,:] = sum_j w[t,j] * FFN_{ids[t,j]}(x[t]) (+ FFN_shared(x[t]))
 * with t = tokens[n].  w13_ptrs[e] / w2_ptrs[e] point at expert e's [2I,H] /
 * [H,I] bf16 blocks (only experts the listed tokens select are read).
 * w13_shared / w2_shared may be NULL.  Tokens are independent (dropless), so
 * this is the same as evaluating the whole batch and keeping those rows.
 */
void oracle_layer_tokens(const uint16_t *x, int64_t H, int64_t I, int64_t k, const int32_t *ids,
                         const double *w, const uint16_t *const *w13_ptrs,
                         const uint16_t *const *w2_ptrs, const uint16_t *w13_shared,
                         const uint16_t *w2_shared, const int64_t *tokens, int64_t n_tokens,
                         double *y, int nthreads) {
#ifdef _OPENMP
#pragma omp parallel for num_threads(nthreads > 0 ? nthreads : 1) schedule(dynamic, 1)
#endif
    for (int64_t n = 0; n < n_tokens; ++n) {
        const int64_t t = tokens[n];
        double *yn = y + n * H;
        double *o = (double *)malloc((size_t)H * sizeof(double));
        for (int64_t c = 0; c < H; ++c) yn[c] = 0.0;
        for (int64_t j = 0; j < k; ++j) {
            const int32_t e = ids[t * k + j];
            oracle_expert_ffn(x + t * H, w13_ptrs[e], w2_ptrs[e], H, I, o);
            for (int64_t c = 0; c < H; ++c) yn[c] += w[t * k + j] * o[c];
        }
        if (w13_shared != NULL && w2_shared != NULL) {
            oracle_expert_ffn(x + t * H, w13_shared, w2_shared, H, I, o);
            for (int64_t c = 0; c < H; ++c) yn[c] += o[c];
        }
        free(o);
    }
    (void)nthreads;
}

/* ---------------------------------------------------- FP8 expert weights --
 * "MoE推理优化全景指南", section "量化与 offload 并非独立开关", "专家权重量化".
 * E4M3 codes with one power-of-two scale per 128 x 128 block: s = the
 * smallest integer with max|w| / 2^s <= 448 (0 for an all-zero block),
 * clamped to [-15, 7] so that code * 2^s is exact in fp16, code
 * = the E4M3 value nearest to w / 2^s (ties to the even code, saturating at
 * 448).  In the binade [2^e, 2^(e+1)) with e >= -6 the E4M3 values are
 * 2^e * (1 + m/8), code (e + 7) * 8 + m; below 2^-6 they are m * 2^-9, code
 * m; rounding m up to 8 lands on the next binade's first code.  nearbyint
 * rounds half to even under the default rounding mode. */
static uint8_t oracle_e4m3(double v) {
  double a = fabs(v);
  if (a > 448.0) a = 448.0;
  int64_t code;
  if (a < ldexp(1.0, -6)) {
    code = (int64_t)nearbyint(ldexp(a, 9));
  } else {
    int x;
    frexp(a, &x); /* a = f * 2^x, f in [0.5, 1) */
    const int e = x - 1;
    code = (int64_t)(e + 7) * 8 + (int64_t)nearbyint((ldexp(a, -e) - 1.0) * 8.0);
  }
  if (code > 0x7E) code = 0x7E;
  if (signbit(v)) code |= 0x80;
  return (uint8_t)code;
}

void oracle_quantize_fp8(const uint16_t *w, int64_t n, int64_t rows, int64_t K, uint8_t *q,
                         int8_t *scale, int nthreads) {
  const int64_t B = 128;
  const int64_t nr = (rows + B - 1) / B, nk = (K + B - 1) / B;
  const int64_t nblocks = n * nr * nk;
#pragma omp parallel for num_threads(nthreads > 0 ? nthreads : 1) schedule(dynamic, 16)
  for (int64_t b = 0; b < nblocks; ++b) {
    const int64_t c = b % nk, r = (b / nk) % nr, i = b / (nk * nr);
    const int64_t r0 = r * B, c0 = c * B;
    const int64_t r1 = r0 + B < rows ? r0 + B : rows, c1 = c0 + B < K ? c0 + B : K;
    double amax = 0.0;
    for (int64_t rr = r0; rr < r1; ++rr)
      for (int64_t cc = c0; cc < c1; ++cc) {
        const double v = fabs(bf16_value(w[(i * rows + rr) * K + cc]));
        if (v > amax) amax = v;
      }
    int s = 0;
    if (amax > 0.0) {
      int x;
      frexp(amax, &x);
      s = x - 9;
      while (ldexp(amax, -s) > 448.0) ++s;
      while (ldexp(amax, -(s - 1)) <= 448.0) --s;
    }
    if (s < -15) s = -15; /* code * 2^s exact in fp16 */
    if (s > 7) s = 7;
    scale[b] = (int8_t)s;
    for (int64_t rr = r0; rr < r1; ++rr)
      for (int64_t cc = c0; cc < c1; ++cc) {
        const int64_t idx = (i * rows + rr) * K + cc;
        q[idx] = oracle_e4m3(ldexp(bf16_value(w[idx]), -s));
      }
  }
}
