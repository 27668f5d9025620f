/*
 * moe_oracle.c -- plain, slow CPU oracle of the single-GPU Mixture-of-Experts
 * layer forward (router -> align -> expert FFN -> weighted combine).
 *
 * TEST INFRASTRUCTURE ONLY.  The tests, the smoke check and the benchmark's
 * CPU-baseline leg are the only code that loads this library.  The CUDA
 * library of the package never links, loads or calls it, and the two share no
 * code, header, table or helper: this file decodes its own input formats and
 * writes every step out in double precision.
 *
 * Sources (web pages; section / figure / equation named per function):
 *   [P1] "How an MoE Model Picks Its Experts During LLM Inference"
 *   [P2] "Mixture of Experts"
 *   [P3] "MoE Kernels, in depth"
 *   [P4] "How GPUs Fuse Communication and Computation During LLM Inference"
 *
 * Pins: every function here is checked by the CPU tests against values the
 * pages print (P1 Figures 1 and 3, the P2 moe_align_block_size worked example),
 * closed forms, brute force on tiny inputs and library casts.  The whole-layer
 * composition has no printed end-to-end value on the pages; it is pinned by
 * hand-derived closed-form layers (logits ln of rationals, SwiGLU at +-ln 3).
 *
 * Conventions shared with the callers (plain C, no CUDA):
 *   dtype codes 0 = bf16, 1 = f32, 2 = FP8 e4m3 (+ one UE8M0 scale byte per 32
 *   consecutive values of a row), 3 = FP4 e2m1 packed two per byte, low nibble
 *   first (+ one UE8M0 scale byte per 32 values of a row).
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define ORC_BF16 0
#define ORC_F32 1
#define ORC_E4M3 2
#define ORC_E2M1 3

/* ------------------------------------------------------------------------ */
/* Number formats.                                                          */
/* ------------------------------------------------------------------------ */

/* bf16 is the upper half of an IEEE binary32. */
double orc_bf16_to_double(uint16_t b) {
  uint32_t u = ((uint32_t)b) << 16;
  float f;
  memcpy(&f, &u, 4);
  return (double)f;
}

/* OCP FP8 E4M3 ("fn": no infinities, S.1111.111 is NaN), exponent bias 7. */
double orc_e4m3_to_double(uint8_t c) {
  int sign = (c >> 7) & 1;
  int e = (c >> 3) & 0xF;
  int m = c & 7;
  double v;
  if (e == 15 && m == 7) return NAN;
  if (e == 0)
    v = ldexp((double)m, -9); /* subnormal: m/8 * 2^(1-7) */
  else
    v = ldexp(1.0 + m / 8.0, e - 7);
  return sign ? -v : v;
}

/* OCP FP4 E2M1: sign, 2 exponent bits (bias 1), 1 mantissa bit. */
double orc_e2m1_to_double(uint8_t nib) {
  int sign = (nib >> 3) & 1;
  int e = (nib >> 1) & 3;
  int m = nib & 1;
  double v = (e == 0) ? 0.5 * m : ldexp(1.0 + 0.5 * m, e - 1);
  return sign ? -v : v;
}

/* UE8M0 block scale: 2^(s-127); 255 is NaN. */
double orc_ue8m0_to_double(uint8_t s) {
  if (s == 255) return NAN;
  return ldexp(1.0, (int)s - 127);
}

/* Round a double to the nearest bf16 value (ties to even); used only by the
 * diagnostic "emulate" mode of the FFN. */
double orc_round_bf16(double v) {
  if (v == 0.0 || isnan(v) || isinf(v)) return v;
  int e;
  frexp(v, &e); /* |v| in [2^(e-1), 2^e) */
  double spacing = ldexp(1.0, e - 8);
  return nearbyint(v / spacing) * spacing;
}

/* Round a double to the nearest e4m3 value (ties to even), saturating at
 * +-448, the largest finite e4m3 value. */
double orc_round_e4m3(double v) {
  if (v == 0.0 || isnan(v)) return v;
  double a = fabs(v), q;
  if (a < ldexp(1.0, -6)) {
    q = nearbyint(a / ldexp(1.0, -9)) * ldexp(1.0, -9);
  } else {
    int e;
    frexp(a, &e); /* a in [2^(e-1), 2^e): 3 mantissa bits -> spacing 2^(e-4) */
    double spacing = ldexp(1.0, e - 4);
    q = nearbyint(a / spacing) * spacing;
  }
  if (q > 448.0) q = 448.0;
  return v < 0 ? -q : q;
}

/* Value of element (row, col) of a row-major matrix with `cols` logical
 * columns stored in `dtype` (scales: one byte per 32 columns of a row). */
static double elem(const void* src, int dtype, const uint8_t* scale, int64_t row,
                   int64_t cols, int64_t col) {
  int64_t i = row * cols + col;
  switch (dtype) {
    case ORC_BF16:
      return orc_bf16_to_double(((const uint16_t*)src)[i]);
    case ORC_F32:
      return (double)((const float*)src)[i];
    case ORC_E4M3: {
      double s = scale ? orc_ue8m0_to_double(scale[row * (cols / 32) + col / 32]) : 1.0;
      return orc_e4m3_to_double(((const uint8_t*)src)[i]) * s;
    }
    case ORC_E2M1: {
      uint8_t byte = ((const uint8_t*)src)[i >> 1];
      uint8_t nib = (i & 1) ? (byte >> 4) : (byte & 15);
      double s = scale ? orc_ue8m0_to_double(scale[row * (cols / 32) + col / 32]) : 1.0;
      return orc_e2m1_to_double(nib) * s;
    }
  }
  return NAN;
}

/* Decode rows [row0, row0+nrows) of a matrix into doubles. */
void orc_decode(const void* src, int dtype, const uint8_t* scale, int64_t row0,
                int64_t nrows, int64_t cols, double* dst) {
  for (int64_t r = 0; r < nrows; ++r)
    for (int64_t c = 0; c < cols; ++c) dst[r * cols + c] = elem(src, dtype, scale, row0 + r, cols, c);
}

/* ------------------------------------------------------------------------ */
/* Router.                                                                  */
/* [P1] Section 1 "What the Router Computes" (three steps; rank key = score */
/* + bias, weight = unbiased score, Figure 3), Section 4 (the five-line     */
/* reference: sigmoid, top-k of score + bias, gather, divide by sum+1e-20), */
/* Section 5.3 (k rounds, lowest id wins ties); Section 1.3 (DeepSeek-V4    */
/* scores with the square root of a softplus instead of a sigmoid).         */
/* [P2] "Mixture of Experts", the gate and DeepSeek's grouped, bias-        */
/* corrected routing (group score = sum of the two largest rank keys of the */
/* group; keep topk_group groups; mask the rest to -inf; top-k; weights     */
/* from the original scores; renormalise; routed scaling factor).           */
/* ------------------------------------------------------------------------ */

/* "a beats b": larger key, ties to the lower id. */
static int beats(double ka, int ia, double kb, int ib) {
  return ka > kb || (ka == kb && ia < ib);
}

/* Router for the listed tokens (all tokens when token_list is NULL).
 *   scoring 0 = softmax over all E logits, 1 = sigmoid per expert,
 *   2 = sqrt(softplus(l)) = sqrt(ln(1 + e^l)) per expert.
 *   n_group <= 1 means plain top-k.
 * Outputs, per listed token i (row i of the outputs):
 *   ids[i*k + j], weights[i*k + j] in selection order (best first);
 *   logits_out[i*E + e] (optional); gap[i] (optional): the margin at the cut,
 *   min(key_k - key_{k+1} over eligible experts, G_(topk_group) -
 *   G_(topk_group+1)), +inf where no competitor exists.
 * Returns 0, or -1 on invalid arguments. */
int orc_router(const void* x, int x_dt, const uint8_t* x_scale, const void* gate, int gate_dt,
               const float* bias, int T, int H, int E, int k, int scoring, int n_group,
               int topk_group, int renormalize, double scaling, const int32_t* token_list,
               int n_tokens, int32_t* ids, double* weights, double* logits_out, double* gap) {
  if (k < 1 || k > E || H < 1 || scoring < 0 || scoring > 2) return -1;
  if (n_group > 1 && (E % n_group != 0 || E / n_group < 2 || topk_group < 1 ||
                      topk_group > n_group || topk_group * (E / n_group) < k))
    return -1;
  int nt = token_list ? n_tokens : T;
  int ret = 0;
#pragma omp parallel for schedule(dynamic, 1)
  for (int i = 0; i < nt; ++i) {
    int t = token_list ? token_list[i] : i;
    if (t < 0 || t >= T) {
      ret = -1;
      continue;
    }
    double* l = (double*)malloc(sizeof(double) * E);
    double* s = (double*)malloc(sizeof(double) * E);
    double* r = (double*)malloc(sizeof(double) * E);
    int* elig = (int*)malloc(sizeof(int) * E);
    double* xr = (double*)malloc(sizeof(double) * H);
    orc_decode(x, x_dt, x_scale, t, 1, H, xr);
    /* Step 1: logits = hidden . gate^T (no bias term in the gate linear). */
    for (int e = 0; e < E; ++e) {
      double acc = 0.0;
      for (int h = 0; h < H; ++h) acc += xr[h] * elem(gate, gate_dt, NULL, e, H, h);
      l[e] = acc;
    }
    if (logits_out) memcpy(logits_out + (int64_t)i * E, l, sizeof(double) * E);
    /* Step 2: scores. */
    if (scoring == 0) {
      double mx = l[0];
      for (int e = 1; e < E; ++e)
        if (l[e] > mx) mx = l[e];
      double sum = 0.0;
      for (int e = 0; e < E; ++e) {
        s[e] = exp(l[e] - mx);
        sum += s[e];
      }
      for (int e = 0; e < E; ++e) s[e] /= sum;
    } else if (scoring == 1) {
      for (int e = 0; e < E; ++e) s[e] = 1.0 / (1.0 + exp(-l[e]));
    } else {
      /* softplus written so that neither exponential overflows */
      for (int e = 0; e < E; ++e) {
        const double sp = l[e] > 0.0 ? l[e] + log1p(exp(-l[e])) : log1p(exp(l[e]));
        s[e] = sqrt(sp);
      }
    }
    /* Rank key: score + selection bias (selection only). */
    for (int e = 0; e < E; ++e) {
      r[e] = s[e] + (bias ? (double)bias[e] : 0.0);
      elig[e] = 1;
    }
    double group_gap = INFINITY;
    if (n_group > 1) {
      int gs = E / n_group;
      double* G = (double*)malloc(sizeof(double) * n_group);
      int* kept = (int*)calloc(n_group, sizeof(int));
      for (int g = 0; g < n_group; ++g) {
        /* sum of the two largest keys of the group */
        double b1 = -INFINITY, b2 = -INFINITY;
        for (int e = g * gs; e < (g + 1) * gs; ++e) {
          if (r[e] > b1) {
            b2 = b1;
            b1 = r[e];
          } else if (r[e] > b2) {
            b2 = r[e];
          }
        }
        G[g] = b1 + b2;
      }
      double last_kept = 0.0;
      for (int round = 0; round < topk_group; ++round) {
        int best = -1;
        for (int g = 0; g < n_group; ++g)
          if (!kept[g] && (best < 0 || beats(G[g], g, G[best], best))) best = g;
        kept[best] = 1;
        last_kept = G[best];
      }
      int first_out = -1;
      for (int g = 0; g < n_group; ++g)
        if (!kept[g] && (first_out < 0 || beats(G[g], g, G[first_out], first_out))) first_out = g;
      if (first_out >= 0) group_gap = last_kept - G[first_out];
      for (int e = 0; e < E; ++e) elig[e] = kept[e / gs];
      free(G);
      free(kept);
    }
    /* Step 3: top-k by rank key, lowest id on ties, k rounds. */
    int* taken = (int*)calloc(E, sizeof(int));
    double wsum = 0.0, kth = 0.0;
    for (int j = 0; j < k; ++j) {
      int best = -1;
      for (int e = 0; e < E; ++e)
        if (elig[e] && !taken[e] && (best < 0 || beats(r[e], e, r[best], best))) best = e;
      taken[best] = 1;
      ids[(int64_t)i * k + j] = best;
      weights[(int64_t)i * k + j] = s[best]; /* the unbiased score */
      wsum += s[best];
      kth = r[best];
    }
    if (gap) {
      int nxt = -1;
      for (int e = 0; e < E; ++e)
        if (elig[e] && !taken[e] && (nxt < 0 || beats(r[e], e, r[nxt], nxt))) nxt = e;
      double g = (nxt >= 0) ? kth - r[nxt] : INFINITY;
      gap[i] = g < group_gap ? g : group_gap;
    }
    for (int j = 0; j < k; ++j) {
      double w = weights[(int64_t)i * k + j];
      if (renormalize) w = w / (wsum + 1e-20);
      weights[(int64_t)i * k + j] = w * scaling;
    }
    free(taken);
    free(l);
    free(s);
    free(r);
    free(elig);
    free(xr);
  }
  return ret;
}

/* ------------------------------------------------------------------------ */
/* Align.  [P3] "Alignment: making ragged routing tileable" (count per      */
/* expert, round each count up to BLOCK_M, exclusive cumulative sum for the */
/* padded starts, assignments of one expert in ascending assignment id,    */
/* padding marked with the sentinel T*k, expert id of every block, padded  */
/* length; buffers sized for the worst case T*k + E*(BLOCK_M-1)).          */
/* [P2] "vLLM's Triton path: align, then index" (the worked example; unused */
/* block entries up to the maximum number of blocks are -1).               */
/* ------------------------------------------------------------------------ */

/* Returns 0; -1 on invalid arguments (an expert id outside [0,E), or a
 * capacity below the worst case). cap_rows entries of sorted_ids and
 * ceil(cap_rows / block_m) entries of block_expert are written. */
int orc_align(const int32_t* topk_ids, int T, int k, int E, int block_m, int64_t cap_rows,
              int32_t* sorted_ids, int32_t* block_expert, int32_t* num_post_padded) {
  int64_t n = (int64_t)T * k;
  if (block_m < 1 || E < 1) return -1;
  if (cap_rows < n + (int64_t)E * (block_m - 1)) return -1;
  for (int64_t a = 0; a < n; ++a)
    if (topk_ids[a] < 0 || topk_ids[a] >= E) return -1;
  int64_t* count = (int64_t*)calloc(E, sizeof(int64_t));
  int64_t* padded = (int64_t*)calloc(E, sizeof(int64_t));
  int64_t* start = (int64_t*)calloc(E, sizeof(int64_t));
  int64_t* placed = (int64_t*)calloc(E, sizeof(int64_t));
  for (int64_t a = 0; a < n; ++a) count[topk_ids[a]]++;
  int64_t total = 0;
  for (int e = 0; e < E; ++e) {
    padded[e] = (count[e] + block_m - 1) / block_m * block_m;
    start[e] = total; /* exclusive cumulative sum */
    total += padded[e];
  }
  int64_t nblocks_cap = (cap_rows + block_m - 1) / block_m;
  for (int64_t p = 0; p < cap_rows; ++p) sorted_ids[p] = (int32_t)n; /* sentinel */
  for (int64_t b = 0; b < nblocks_cap; ++b) block_expert[b] = -1;
  /* Visiting assignments in ascending id keeps each expert's run in
   * ascending assignment order (a stable sort by expert). */
  for (int64_t a = 0; a < n; ++a) {
    int e = topk_ids[a];
    sorted_ids[start[e] + placed[e]] = (int32_t)a;
    placed[e]++;
  }
  for (int e = 0; e < E; ++e)
    for (int64_t b = start[e] / block_m; b < (start[e] + padded[e]) / block_m; ++b) block_expert[b] = e;
  *num_post_padded = (int32_t)total;
  free(count);
  free(padded);
  free(start);
  free(placed);
  return 0;
}

/* ------------------------------------------------------------------------ */
/* Expert FFN and combine.                                                  */
/* [P3] "The kernel inventory of one layer": the naive per-expert loop      */
/* y[idx_e] += w_e * ffn_e(x[idx_e]) is the reference; "The fused expert    */
/* GEMM": gate and up stored as one 2F x H matrix, SwiGLU silu(g) * u.      */
/* [P2] "Mixture of Experts": w13 [E, 2F, H] (gate rows first, then up      */
/* rows), w2 [E, H, F].  [P4] Section 1.1: SwiGLU silu(gate) * up, second   */
/* multiplication back to H, sum of the k outputs times their weights;      */
/* Section 3.5: FP8 re-quantisation with a power-of-two scale per 32 values */
/* (scale = smallest power of two >= amax / 448).                           */
/* ------------------------------------------------------------------------ */

static double silu(double z) { return z / (1.0 + exp(-z)); }

/* One expert applied to one hidden row: out[H] = W2[e] (silu(G x) * (U x)).
 * emulate: 0 exact; 1 round the activation to bf16; 2 re-quantise the
 * activation to e4m3 with a UE8M0 scale per 32 values. */
void orc_expert_ffn(const double* xr, const void* w13, const uint8_t* w13_scale, const void* w2,
                    const uint8_t* w2_scale, int w_dt, int H, int F, int e, int emulate,
                    double* out) {
  double* hbuf = (double*)malloc(sizeof(double) * 2 * F);
  double* act = (double*)malloc(sizeof(double) * F);
  double* wrow = (double*)malloc(sizeof(double) * (H > F ? H : F));
  for (int i = 0; i < 2 * F; ++i) {
    orc_decode(w13, w_dt, w13_scale, (int64_t)e * 2 * F + i, 1, H, wrow);
    double acc = 0.0;
    for (int h = 0; h < H; ++h) acc += wrow[h] * xr[h];
    hbuf[i] = acc;
  }
  for (int f = 0; f < F; ++f) act[f] = silu(hbuf[f]) * hbuf[F + f];
  if (emulate == 1) {
    for (int f = 0; f < F; ++f) act[f] = orc_round_bf16(act[f]);
  } else if (emulate == 2) {
    for (int f0 = 0; f0 < F; f0 += 32) {
      double amax = 0.0;
      for (int f = f0; f < f0 + 32 && f < F; ++f)
        if (fabs(act[f]) > amax) amax = fabs(act[f]);
      double scale = 1.0;
      if (amax > 0.0) scale = ldexp(1.0, (int)ceil(log2(amax / 448.0)));
      for (int f = f0; f < f0 + 32 && f < F; ++f) act[f] = orc_round_e4m3(act[f] / scale) * scale;
    }
  }
  for (int h = 0; h < H; ++h) {
    orc_decode(w2, w_dt, w2_scale, (int64_t)e * H + h, 1, F, wrow);
    double acc = 0.0;
    for (int f = 0; f < F; ++f) acc += wrow[f] * act[f];
    out[h] = acc;
  }
  free(hbuf);
  free(act);
  free(wrow);
}

/* Layer output for the listed tokens (all tokens when token_list is NULL),
 * given the routing (ids, weights: [T, k]).  Per token, contributions are
 * added in ascending expert id, the order of the naive per-expert loop.
 * y: [n_listed, H].  emulate 1/2 additionally round each weighted expert
 * output to bf16 before the sum (the staging precision of the GPU path). */
int orc_moe_ffn(const void* x, int x_dt, const uint8_t* x_scale, const void* w13,
                const uint8_t* w13_scale, const void* w2, const uint8_t* w2_scale, int w_dt, int T,
                int H, int F, int E, int k, const int32_t* ids, const double* weights,
                const int32_t* token_list, int n_tokens, int emulate, double* y) {
  int nt = token_list ? n_tokens : T;
  int ret = 0;
#pragma omp parallel for schedule(dynamic, 1)
  for (int i = 0; i < nt; ++i) {
    int t = token_list ? token_list[i] : i;
    if (t < 0 || t >= T) {
      ret = -1;
      continue;
    }
    double* xr = (double*)malloc(sizeof(double) * H);
    double* o = (double*)malloc(sizeof(double) * H);
    double* yr = y + (int64_t)i * H;
    orc_decode(x, x_dt, x_scale, t, 1, H, xr);
    for (int h = 0; h < H; ++h) yr[h] = 0.0;
    for (int e = 0; e < E; ++e) {
      for (int j = 0; j < k; ++j) {
        if (ids[(int64_t)t * k + j] != e) continue;
        double w = weights[(int64_t)t * k + j];
        orc_expert_ffn(xr, w13, w13_scale, w2, w2_scale, w_dt, H, F, e, emulate, o);
        for (int h = 0; h < H; ++h) {
          double c = w * o[h];
          if (emulate) c = orc_round_bf16(c);
          yr[h] += c;
        }
      }
    }
    free(xr);
    free(o);
  }
  return ret;
}

/* Number of threads OpenMP would use (for reporting). */
/* ------------------------------------------------------------------------ */
/* FP8 cast of the layer input.                                             */
/* "How GPUs Fuse Communication and Computation During LLM Inference" §1.1  */
/* (a small cast kernel turns the layer input into FP8 codes and writes the */
/* scales) with the scale rule of §3.5 (per 32 values, the smallest power   */
/* of two 2^s with amax / 2^s <= 448; codes = e4m3(value / 2^s), nearest,   */
/* ties to even, saturating); "MoE Kernels, in depth", Low precision (the   */
/* activation quantisation belongs in a pass that moves the rows anyway).   */
/* ------------------------------------------------------------------------ */

/* e4m3 code of a value that is already an e4m3 value (or +-0): the code in
 * the 256-entry table whose value it is (sign from the sign bit, so -0 is
 * 0x80).  Returns 0xFF (a NaN code) if there is none. */
static uint8_t e4m3_code_of(double q) {
  const int neg = signbit(q) ? 1 : 0;
  const double a = fabs(q);
  for (int c = 0; c < 128; ++c)
    if (c != 0x7F && orc_e4m3_to_double((uint8_t)c) == a) return (uint8_t)(c | (neg << 7));
  return 0xFF;
}

/* codes [T*H] and scale bytes [T*H/32] of x [T,H] (bf16 or f32), H % 32 == 0.
 * s is found by stepping from -127 (the smallest UE8M0 exponent) upward, so it
 * is the smallest s in [-127, 127] with amax <= 448 * 2^s (s = 0 for an
 * all-zero group).  Returns 0, or -1 on invalid arguments. */
int orc_quantize_e4m3(const void* x, int x_dt, int T, int H, uint8_t* codes, uint8_t* scales) {
  if (T < 0 || H <= 0 || H % 32 != 0 || (x_dt != 0 && x_dt != 1)) return -1;
  int bad = 0;
#pragma omp parallel for schedule(static)
  for (int t = 0; t < T; ++t) {
    for (int g = 0; g < H / 32; ++g) {
      double v[32], amax = 0.0;
      for (int i = 0; i < 32; ++i) {
        v[i] = elem(x, x_dt, NULL, t, H, g * 32 + i);
        if (fabs(v[i]) > amax) amax = fabs(v[i]);
      }
      int s = 0;
      if (amax > 0.0) {
        s = -127;
        while (s < 127 && amax > 448.0 * ldexp(1.0, s)) ++s;
      }
      scales[(int64_t)t * (H / 32) + g] = (uint8_t)(s + 127);
      for (int i = 0; i < 32; ++i) {
        const uint8_t c = e4m3_code_of(orc_round_e4m3(v[i] / ldexp(1.0, s)));
        if (c == 0xFF) bad = 1;
        codes[(int64_t)t * H + g * 32 + i] = c;
      }
    }
  }
  return bad ? -1 : 0;
}

int orc_num_threads(void) {
#ifdef _OPENMP
  extern int omp_get_max_threads(void);
  return omp_get_max_threads();
#else
  return 1;
#endif
}
