/*
 * oracle.c -- plain, slow, obviously-correct CPU oracle for the fused MoE forward pass.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the product path may call, link or load this file:
 * only the tests, the smoke check of the package entry module and the cpu_baseline leg of
 * the benchmark use it.  It shares no code, header, table or constant generator with the
 * CUDA library.
 *
 * What it computes (sources are the four web pages the project is built from):
 *   - TileOPs benchmark page, "MoE" section, op FusedMoEFwd: hidden_states[T,H],
 *     gating_output[T,E] f32, w_gate_up[E,2F,H], w_down[E,H,F], top_k, renormalize; the
 *     sigmoid variant adds correction_bias[E] f32, num_expert_group, topk_group and
 *     routed_scaling_factor.  Op FusedMoESharedExpertFwd adds shared_w_gate_up[2S,H] and
 *     shared_w_down[H,S].  Op MoEGroupedGemmFwd names the activation silu_and_mul.
 *   - The same page's ops FusedTopKFwd (router), MoEPermuteAlignFwd (sort),
 *     MoEPostPermuteFwd (weighted combine of expert rows through inverse indices).
 *   - flashinfer PR #4048 (CuTe DSL W4A16 MoE) and its weight-scale placement ablation: NVFP4
 *     experts, E2M1 codes with E4M3 block scales over 16 elements and an FP32 per-expert scale
 *     (oracle_moe_tokens_w4 and the stage references after it).
 *   - The same page's op MoEGroupedGemmFP8Fwd: E4M3 operands with f32 scales per 128-k block of
 *     a row and per 128 x 128 block of weights (oracle_grouped_gemm_fp8).
 *   - The same page's op MoEGroupedGemmFwd in its contiguous and masked layouts
 *     (oracle_grouped_gemm) and op MoEPostPermuteFwd with route weights (oracle_post_permute).
 *   - ROCm/aiter PR #5973 "[FlyDSL] Optimize MI308 MoE decoding (3/3)", section "Changes":
 *     routes whose expert id is -1 are padding and are skipped; the prefill sort returns each
 *     route's sorted row (the inverse map produced here).
 *
 * Precision: every floating-point step is fp64 over the bf16/f16-rounded inputs, except the
 * one place where floating point decides an integer.  The sigmoid routing key that decides
 * which experts are selected is evaluated in f32 (the precision of gating_output) by a fixed
 * sequence of correctly rounded operations, so that selection is reproducible bit for bit; see
 * oracle_sigmoid_key_f32.
 *
 * Parity pins (tests/test_oracle_pins.py): brute-force routing on tiny inputs, weight sum
 * invariants, E=1/top_k=1 reduction to a dense SwiGLU MLP computed by a textbook matvec, the
 * GeGLU-tanh activation against the exact GELU x*Phi(x) within the tanh form's error, ReLU2
 * against max(g,0)^2 on every sign,
 * token-permutation equivariance, zeroed-expert and linearity checks, sort invariants, the
 * bf16/f16 decoders against every bit pattern, and the f32 exp/sigmoid against fp64 within
 * stated ulp bounds.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define ORACLE_OK 0
#define ORACLE_ERR_ARG 1
#define ORACLE_ERR_ID 6

/* ------------------------------------------------------------------------------------------ */
/* 16-bit float decoding, written from the IEEE 754 binary16 and bfloat16 definitions.         */
/* ------------------------------------------------------------------------------------------ */

/* bfloat16: the upper 16 bits of an IEEE binary32. */
static double bf16_bits_to_double(uint16_t b) {
  uint32_t u = ((uint32_t)b) << 16;
  float f;
  memcpy(&f, &u, sizeof f);
  return (double)f;
}

/* IEEE binary16: 1 sign bit, 5 exponent bits (bias 15), 10 fraction bits. */
static double f16_bits_to_double(uint16_t b) {
  int sign = (b >> 15) & 1;
  int ex = (b >> 10) & 0x1f;
  int fr = b & 0x3ff;
  double v;
  if (ex == 0) {
    v = ldexp((double)fr, -24); /* subnormal: fr * 2^-14 * 2^-10 */
  } else if (ex == 31) {
    v = fr ? NAN : INFINITY;
  } else {
    v = ldexp((double)(1024 + fr), ex - 25); /* (1 + fr/1024) * 2^(ex-15) */
  }
  return sign ? -v : v;
}

double oracle_half_bits_to_double(int dtype, uint16_t bits) {
  return dtype == 0 ? bf16_bits_to_double(bits) : f16_bits_to_double(bits);
}

void oracle_decode_array(int dtype, const uint16_t* in, double* out, int64_t n) {
  for (int64_t i = 0; i < n; ++i) out[i] = oracle_half_bits_to_double(dtype, in[i]);
}

/* One lookup table per dtype: decoding is a pure function of the 16 bits. */
static double g_tab[2][65536];
static int g_tab_ready[2];

static const double* decode_table(int dtype) {
  if (!g_tab_ready[dtype]) {
    for (int i = 0; i < 65536; ++i) g_tab[dtype][i] = oracle_half_bits_to_double(dtype, (uint16_t)i);
    g_tab_ready[dtype] = 1;
  }
  return g_tab[dtype];
}

/* ------------------------------------------------------------------------------------------ */
/* f32 routing key for scoring_func=sigmoid.                                                   */
/*                                                                                            */
/* The pages give gating_output in f32 and select experts on sigmoid scores plus the f32       */
/* correction_bias; they fix no formula for the f32 sigmoid.  Selection is an integer result   */
/* decided by floating point, so it is taken in f32 (the kernel's precision), and the f32      */
/* sigmoid is defined here as an explicit sequence of IEEE-754 correctly rounded operations:   */
/*   z = clamp(-x, -80, 80)                                                                    */
/*   exp(z) by Cody-Waite range reduction: n = rint(z * log2(e)), r = z - n*ln2 (ln2 split     */
/*   into a 16-bit head and an f32 tail), exp(r) by the degree-7 Taylor polynomial of e^r      */
/*   (coefficients 1/k!) evaluated by Horner's rule with fused multiply-adds, times 2^n;        */
/*   sigmoid = 1 / (1 + exp(z)).                                                                */
/* The polynomial remainder is below 1e-8 relative for |r| <= ln2/2, so the result is within   */
/* a few f32 ulps of the true sigmoid (pinned by the tests against fp64).                       */
/* ------------------------------------------------------------------------------------------ */
static const float K_LOG2E = 0x1.715476p+0f;  /* log2(e) rounded to f32 */
static const float K_LN2_HI = 0x1.62e4p-1f;   /* 45426 / 65536: ln 2 to 16 bits, n*HI exact */
static const float K_LN2_LO = 0x1.7f7d1cp-20f; /* ln 2 - K_LN2_HI rounded to f32 */
static const float K_C2 = 0x1p-1f;            /* 1/2! */
static const float K_C3 = 0x1.555556p-3f;     /* 1/3! */
static const float K_C4 = 0x1.555556p-5f;     /* 1/4! */
static const float K_C5 = 0x1.111112p-7f;     /* 1/5! */
static const float K_C6 = 0x1.6c16c2p-10f;    /* 1/6! */
static const float K_C7 = 0x1.a01a02p-13f;    /* 1/7! */

float oracle_exp_f32(float z) {
  float n = rintf(z * K_LOG2E);
  float r = fmaf(-n, K_LN2_HI, z);
  r = fmaf(-n, K_LN2_LO, r);
  float p = K_C7;
  p = fmaf(p, r, K_C6);
  p = fmaf(p, r, K_C5);
  p = fmaf(p, r, K_C4);
  p = fmaf(p, r, K_C3);
  p = fmaf(p, r, K_C2);
  p = fmaf(p, r, 1.0f);
  p = fmaf(p, r, 1.0f);
  int ni = (int)n; /* |n| <= 116 for |z| <= 80, so 2^n is a normal f32 */
  uint32_t bits = (uint32_t)(ni + 127) << 23;
  float two_n;
  memcpy(&two_n, &bits, sizeof two_n);
  return p * two_n;
}

float oracle_sigmoid_key_f32(float x) {
  float z = -x;
  z = fminf(fmaxf(z, -80.0f), 80.0f);
  float e = oracle_exp_f32(z);
  return 1.0f / (1.0f + e);
}

/* ------------------------------------------------------------------------------------------ */
/* Router (TileOPs "MoE" page, ops FusedTopKFwd and FusedMoEFwd).                              */
/* ------------------------------------------------------------------------------------------ */

/* a ranks before b: larger key first, equal keys -> lower index first. */
static int ranks_before_f(float ka, int ia, float kb, int ib) {
  return ka > kb || (ka == kb && ia < ib);
}

/* Pick the index of the best remaining entry of keys[0..n) among allowed[]; -1 if none. */
static int pick_best(const float* keys, const unsigned char* allowed, int n) {
  int best = -1;
  for (int i = 0; i < n; ++i) {
    if (!allowed[i]) continue;
    if (best < 0 || ranks_before_f(keys[i], i, keys[best], best)) best = i;
  }
  return best;
}

/*
 * oracle_route: top-k expert ids and weights per token.
 *   scoring 0 (softmax): select the top_k raw logits (softmax is monotone, so this is the same
 *     selection as on probabilities); weight_j = exp(x_j - m) / sum, where the sum runs over the
 *     selected experts if renormalize, else over all E; times routed_scaling_factor.
 *   scoring 1 (sigmoid): s_e = sigmoid(x_e); selection key b_e = s_e + correction_bias_e (f32);
 *     if num_expert_group G > 1: group g holds experts [g*E/G, (g+1)*E/G), its score is the sum
 *     of its two largest keys, the topk_group best groups are kept (ties -> lower group), the
 *     other experts are excluded; the top_k keys among the kept experts are selected (ties ->
 *     lower id); weight_j = s_j / sum_sel(s) if renormalize, else s_j; times rsf.
 * ids are written in selection order (descending key, ties -> lower id).  Weights use the fp64
 * sigmoid of x (the plain definition); only the selection uses the f32 key.
 * near_tie (nullable) gets 1 for a token whose selection boundary gap in the f32 keys is below
 * 1e-6 (a diagnostic only; selection is still decided exactly).
 */
int oracle_route(int T, int E, int top_k, int scoring, int renormalize, int num_expert_group,
                 int topk_group, double rsf, const float* gating, const float* bias, int32_t* ids,
                 double* weights, int32_t* near_tie) {
  if (T < 0 || E <= 0 || top_k <= 0 || top_k > E) return ORACLE_ERR_ARG;
  int G = num_expert_group > 1 ? num_expert_group : 1;
  int keepG = G > 1 ? topk_group : 1;
  if (G > 1 && (scoring != 1 || E % G != 0 || E / G < 2 || keepG < 1 || keepG > G ||
                keepG * (E / G) < top_k))
    return ORACLE_ERR_ARG;
  if (scoring == 0 && bias) return ORACLE_ERR_ARG;
  float* key = (float*)malloc(sizeof(float) * E);
  unsigned char* allowed = (unsigned char*)malloc(E);
  float* gscore = (float*)malloc(sizeof(float) * G);
  unsigned char* gallowed = (unsigned char*)malloc(G);
  unsigned char* gkeep = (unsigned char*)malloc(G);
  for (int t = 0; t < T; ++t) {
    const float* x = gating + (int64_t)t * E;
    int32_t* id_t = ids + (int64_t)t * top_k;
    double* w_t = weights + (int64_t)t * top_k;
    int tie = 0;
    for (int e = 0; e < E; ++e) {
      if (scoring == 0) {
        key[e] = x[e];
      } else {
        float s = oracle_sigmoid_key_f32(x[e]);
        key[e] = bias ? s + bias[e] : s;
      }
      if (key[e] != key[e]) key[e] = -INFINITY; /* a NaN key ranks lowest */
      allowed[e] = 1;
    }
    if (G > 1 && keepG < G) {
      int gs = E / G;
      for (int g = 0; g < G; ++g) {
        /* sum of the two largest keys of the group */
        float m1 = -INFINITY, m2 = -INFINITY;
        for (int i = 0; i < gs; ++i) {
          float v = key[g * gs + i];
          if (v > m1) { m2 = m1; m1 = v; }
          else if (v > m2) { m2 = v; }
        }
        gscore[g] = m1 + m2;
        gallowed[g] = 1;
        gkeep[g] = 0;
      }
      int last = -1;
      for (int j = 0; j < keepG; ++j) {
        int g = pick_best(gscore, gallowed, G);
        gkeep[g] = 1;
        gallowed[g] = 0;
        last = g;
      }
      int next = pick_best(gscore, gallowed, G);
      if (next >= 0 && fabs((double)gscore[last] - (double)gscore[next]) < 1e-6) tie = 1;
      for (int e = 0; e < E; ++e) allowed[e] = gkeep[e / gs];
    }
    for (int j = 0; j < top_k; ++j) {
      int e = pick_best(key, allowed, E);
      id_t[j] = e;
      allowed[e] = 0;
    }
    {
      int next = pick_best(key, allowed, E);
      if (next >= 0 && fabs((double)key[id_t[top_k - 1]] - (double)key[next]) < 1e-6) tie = 1;
    }
    if (near_tie) near_tie[t] = tie;
    /* weights in fp64 */
    if (scoring == 0) {
      double m = -INFINITY;
      for (int e = 0; e < E; ++e) if ((double)x[e] > m) m = x[e];
      double denom = 0.0;
      if (renormalize) {
        for (int j = 0; j < top_k; ++j) denom += exp((double)x[id_t[j]] - m);
      } else {
        for (int e = 0; e < E; ++e) denom += exp((double)x[e] - m);
      }
      for (int j = 0; j < top_k; ++j) w_t[j] = exp((double)x[id_t[j]] - m) / denom * rsf;
    } else {
      double denom = 0.0;
      for (int j = 0; j < top_k; ++j) denom += 1.0 / (1.0 + exp(-(double)x[id_t[j]]));
      for (int j = 0; j < top_k; ++j) {
        double s = 1.0 / (1.0 + exp(-(double)x[id_t[j]]));
        w_t[j] = (renormalize ? s / denom : s) * rsf;
      }
    }
  }
  free(key);
  free(allowed);
  free(gscore);
  free(gallowed);
  free(gkeep);
  return ORACLE_OK;
}

/* a ranks before b in fp64: larger key first, equal keys -> lower index first. */
static int ranks_before_d(double ka, int ia, double kb, int ib) {
  return ka > kb || (ka == kb && ia < ib);
}

static int pick_best_d(const double* keys, const unsigned char* allowed, int n) {
  int best = -1;
  for (int i = 0; i < n; ++i) {
    if (!allowed[i]) continue;
    if (best < 0 || ranks_before_d(keys[i], i, keys[best], best)) best = i;
  }
  return best;
}

/*
 * oracle_route_select_f64: the sigmoid selection of oracle_route taken on the plain definition,
 * every step in fp64 (TileOPs "MoE" page, FusedTopKFwd / FusedMoEFwd parameters scoring_func,
 * correction_bias, num_expert_group, topk_group): s_e = 1 / (1 + exp(-x_e)),
 * b_e = s_e + correction_bias_e; a group's score is the sum of its two largest b; the topk_group
 * best groups are kept (ties -> lower group); the top_k largest b among the kept experts are
 * selected (ties -> lower id), in descending order.  It exists to check the f32 selection key
 * of oracle_route against the definition it approximates.
 * Per token it also returns
 *   boundary_gap  the smallest fp64 gap at a selection boundary: between the last kept and the
 *                 first dropped group score, and between the top_k-th and the next candidate
 *                 key (+inf where there is no such pair).  Below ~1e-6 the f32 keys may
 *                 legitimately choose differently.
 *   order_gap     the smallest gap between consecutive selected keys (+inf for top_k = 1):
 *                 below ~1e-6 the f32 keys may order the same experts differently.
 */
int oracle_route_select_f64(int T, int E, int top_k, int num_expert_group, int topk_group,
                            const float* gating, const float* bias, int32_t* ids,
                            double* boundary_gap, double* order_gap) {
  if (T < 0 || E <= 0 || top_k <= 0 || top_k > E) return ORACLE_ERR_ARG;
  int G = num_expert_group > 1 ? num_expert_group : 1;
  int keepG = G > 1 ? topk_group : 1;
  if (G > 1 && (E % G != 0 || E / G < 2 || keepG < 1 || keepG > G || keepG * (E / G) < top_k))
    return ORACLE_ERR_ARG;
  double* key = (double*)malloc(sizeof(double) * E);
  unsigned char* allowed = (unsigned char*)malloc(E);
  double* gscore = (double*)malloc(sizeof(double) * G);
  unsigned char* gallowed = (unsigned char*)malloc(G);
  unsigned char* gkeep = (unsigned char*)malloc(G);
  for (int t = 0; t < T; ++t) {
    const float* x = gating + (int64_t)t * E;
    int32_t* id_t = ids + (int64_t)t * top_k;
    double bgap = INFINITY, ogap = INFINITY;
    for (int e = 0; e < E; ++e) {
      double sv = 1.0 / (1.0 + exp(-(double)x[e]));
      key[e] = bias ? sv + (double)bias[e] : sv;
      if (key[e] != key[e]) key[e] = -INFINITY; /* a NaN key ranks lowest */
      allowed[e] = 1;
    }
    if (G > 1 && keepG < G) {
      int gs = E / G;
      for (int g = 0; g < G; ++g) {
        double m1 = -INFINITY, m2 = -INFINITY;
        for (int i = 0; i < gs; ++i) {
          double v = key[g * gs + i];
          if (v > m1) { m2 = m1; m1 = v; }
          else if (v > m2) { m2 = v; }
        }
        gscore[g] = m1 + m2;
        gallowed[g] = 1;
        gkeep[g] = 0;
      }
      int last = -1;
      for (int j = 0; j < keepG; ++j) {
        int g = pick_best_d(gscore, gallowed, G);
        gkeep[g] = 1;
        gallowed[g] = 0;
        last = g;
      }
      int next = pick_best_d(gscore, gallowed, G);
      if (next >= 0) bgap = fabs(gscore[last] - gscore[next]);
      for (int e = 0; e < E; ++e) allowed[e] = gkeep[e / gs];
    }
    for (int j = 0; j < top_k; ++j) {
      int e = pick_best_d(key, allowed, E);
      id_t[j] = e;
      allowed[e] = 0;
      if (j > 0) {
        double d = fabs(key[id_t[j - 1]] - key[e]);
        if (d < ogap) ogap = d;
      }
    }
    {
      int next = pick_best_d(key, allowed, E);
      if (next >= 0) {
        double d = fabs(key[id_t[top_k - 1]] - key[next]);
        if (d < bgap) bgap = d;
      }
    }
    if (boundary_gap) boundary_gap[t] = bgap;
    if (order_gap) order_gap[t] = ogap;
  }
  free(key);
  free(allowed);
  free(gscore);
  free(gallowed);
  free(gkeep);
  return ORACLE_OK;
}

/* ------------------------------------------------------------------------------------------ */
/* Expert sort (TileOPs "MoE" page, op MoEPermuteAlignFwd; aiter PR #5973 "Changes": the sort */
/* returns each route's sorted row).  A plain counting sort of flat route indices r = t*k + j. */
/* ------------------------------------------------------------------------------------------ */

/*
 * counts[e]     number of routes with id e (ids of -1 are padding and are skipped)
 * offsets[e]    start of expert e's segment; segments are padded to a multiple of block_m;
 *               offsets[E] is the padded total
 * sorted_ids[p] flat route index at sorted position p, ascending within each segment; -1 in
 *               padding slots and in every slot from offsets[E] to sorted_len
 * tile_expert[i] expert owning rows [i*block_m, (i+1)*block_m); -1 from offsets[E]/block_m on
 * inv_route[r]  sorted position of route r, -1 for a padding route
 * Any id outside [-1, E) returns ORACLE_ERR_ID.
 */
int oracle_align_sort(int T, int top_k, int E, int block_m, const int32_t* ids, int32_t* counts,
                      int32_t* offsets, int32_t* sorted_ids, int64_t sorted_len,
                      int32_t* tile_expert, int64_t tile_len, int32_t* inv_route) {
  if (T < 0 || top_k <= 0 || E <= 0 || block_m <= 0) return ORACLE_ERR_ARG;
  int64_t P = (int64_t)T * top_k;
  for (int64_t r = 0; r < P; ++r)
    if (ids[r] < -1 || ids[r] >= E) return ORACLE_ERR_ID;
  for (int e = 0; e < E; ++e) counts[e] = 0;
  for (int64_t r = 0; r < P; ++r)
    if (ids[r] >= 0) counts[ids[r]] += 1;
  offsets[0] = 0;
  for (int e = 0; e < E; ++e) {
    int padded = (counts[e] + block_m - 1) / block_m * block_m;
    offsets[e + 1] = offsets[e] + padded;
  }
  if (offsets[E] > sorted_len || offsets[E] / block_m > tile_len) return ORACLE_ERR_ARG;
  for (int64_t p = 0; p < sorted_len; ++p) sorted_ids[p] = -1;
  int32_t* fill = (int32_t*)malloc(sizeof(int32_t) * E);
  for (int e = 0; e < E; ++e) fill[e] = offsets[e];
  for (int64_t r = 0; r < P; ++r) {
    int e = ids[r];
    if (e < 0) {
      inv_route[r] = -1;
      continue;
    }
    sorted_ids[fill[e]] = (int32_t)r;
    inv_route[r] = fill[e];
    fill[e] += 1;
  }
  free(fill);
  for (int64_t i = 0; i < tile_len; ++i) tile_expert[i] = -1;
  for (int e = 0; e < E; ++e)
    for (int p = offsets[e]; p < offsets[e + 1]; p += block_m) tile_expert[p / block_m] = e;
  return ORACLE_OK;
}

/* ------------------------------------------------------------------------------------------ */
/* Expert MLP (TileOPs "MoE" page, ops MoEGroupedGemmFwd with activation=silu_and_mul,          */
/* MoEExpertMLPFwd and SharedExpertMLPFwd): rows [0,F) of w_gate_up are the gate, rows [F,2F)   */
/* the up projection; act = SiLU(gate) * up with SiLU(g) = g / (1 + e^-g); y = w_down . act.     */
/* Activation variants (flashinfer PR #4048 follow-up "Extend CuTe DSL W4A16 fused MoE with      */
/* tanh-approximate GeGLU and SiTU", and the W4A8 validation list naming SwiGLU and ReLU2):      */
/*   GeGLU-tanh  act = up * GELU_tanh(gate),                                                     */
/*               GELU_tanh(g) = g/2 * (1 + tanh(sqrt(2/pi) * (g + 0.044715 g^3)));              */
/*   ReLU2       act = max(g, 0)^2 of a single projection: w_gate_up has F rows (no up half).    */
/* ------------------------------------------------------------------------------------------ */

#define ORACLE_ACT_SILU 0
#define ORACLE_ACT_GELU_TANH 1
#define ORACLE_ACT_RELU2 2

/* Rows per expert of w_gate_up: 2F for the gated activations, F for ReLU2. */
static int64_t gate_up_rows(int activation, int F) {
  return activation == ORACLE_ACT_RELU2 ? (int64_t)F : (int64_t)2 * F;
}

static double gelu_tanh(double g) {
  const double c = sqrt(2.0 / 3.14159265358979323846);
  return 0.5 * g * (1.0 + tanh(c * (g + 0.044715 * g * g * g)));
}

/* act[f] for one expert: wgu is [gate_up_rows(activation, F), H]. */
static void act_rows(const double* tab, const uint16_t* wgu, const double* x, int H, int F,
                     int activation, double* act) {
  for (int f = 0; f < F; ++f) {
    const uint16_t* wg = wgu + (int64_t)f * H;
    double g = 0.0;
    for (int h = 0; h < H; ++h) g += tab[wg[h]] * x[h];
    if (activation == ORACLE_ACT_RELU2) {
      const double r = g > 0.0 ? g : 0.0;
      act[f] = r * r;
      continue;
    }
    const uint16_t* wu = wgu + (int64_t)(F + f) * H;
    double u = 0.0;
    for (int h = 0; h < H; ++h) u += tab[wu[h]] * x[h];
    if (activation == ORACLE_ACT_GELU_TANH)
      act[f] = gelu_tanh(g) * u;
    else
      act[f] = g / (1.0 + exp(-g)) * u;
  }
}

/* y[h] = sum_f Wd[h,f] act[f] for one expert; wd is [H, F]. */
static void down_rows(const double* tab, const uint16_t* wd, const double* act, int H, int F,
                      double* y) {
  for (int h = 0; h < H; ++h) {
    const uint16_t* w = wd + (int64_t)h * F;
    double s = 0.0;
    for (int f = 0; f < F; ++f) s += tab[w[f]] * act[f];
    y[h] = s;
  }
}

/* Half the spacing of a 16-bit float type at |a| (dtype 0 bf16: 8 significant bits, 1 f16:
 * 11; below the smallest normal the subnormal spacing): the largest error of rounding a to it. */
static double half_ulp16(int dtype, double a) {
  a = fabs(a);
  if (a == 0.0) return 0.0;
  int ex;
  frexp(a, &ex); /* a = m * 2^ex with m in [0.5, 1): a lies in the binade [2^(ex-1), 2^ex) */
  const int bits = dtype == 0 ? 8 : 11;
  const int emin = dtype == 0 ? -126 : -14;
  const int e = ex - 1 < emin ? emin : ex - 1;
  return ldexp(1.0, e - bits);
}

/* noise[h] += wsq * sum_f (Wd[h,f] * half_ulp16(act[f]))^2: the variance scale of the error that
 * rounding act to the 16-bit type adds to y[h] = Wd . act (each rounding error lies within
 * +-half an ulp of its act value). */
static void down_noise(const double* tab, const uint16_t* wd, const double* act, int H, int F,
                       int dtype, double wsq, double* u, double* noise) {
  for (int f = 0; f < F; ++f) u[f] = half_ulp16(dtype, act[f]);
  for (int h = 0; h < H; ++h) {
    const uint16_t* w = wd + (int64_t)h * F;
    double s = 0.0;
    for (int f = 0; f < F; ++f) {
      const double c = tab[w[f]] * u[f];
      s += c * c;
    }
    noise[h] += wsq * s;
  }
}

/* Expert weights are addressed through slot[e] (identity when slot is NULL) so that a caller
 * can pass only the experts a sampled set of tokens touches. */
static const uint16_t* expert_ptr(const uint16_t* base, const int32_t* slot, int e, int64_t stride) {
  int s = slot ? slot[e] : e;
  if (s < 0) return NULL;
  return base + (int64_t)s * stride;
}

/*
 * oracle_moe_tokens: the fused MoE forward for a list of tokens, per token in fp64:
 *   out[t] = sum_j weights[t,j] * W_down[e_j] . act(x_t; w_gate_up[e_j])
 *            + shared(x_t)            (shared term only when S > 0; unweighted, not scaled)
 * with act() the activation selected by `activation` (ORACLE_ACT_*, see act_rows); the shared
 * expert uses the same activation.
 * Routes with id -1 are skipped.  out is [n_tok, H] in the order of tok_list.
 * act_noise (nullable, [n_tok, H]): per output element
 *   sqrt( sum_j weights[t,j]^2 sum_f (W_down[e_j][h,f] u(act_j[f]))^2 + shared term )
 * with u(a) half an ulp of the 16-bit dtype at a -- the scale of the error a computation that
 * rounds each act value to that dtype before the down projection makes (a diagnostic of the
 * arithmetic; out itself never rounds).
 */
int oracle_moe_tokens(int n_tok, const int32_t* tok_list, int T, int H, int E, int F, int top_k,
                      int dtype, int activation, const uint16_t* hidden, const int32_t* ids,
                      const double* weights, const uint16_t* w_gate_up, const uint16_t* w_down,
                      const int32_t* expert_slot, int S, const uint16_t* shared_w_gate_up,
                      const uint16_t* shared_w_down, double* out, double* act_noise) {
  if (n_tok < 0 || H <= 0 || E <= 0 || F <= 0 || top_k <= 0 || (dtype != 0 && dtype != 1) ||
      activation < ORACLE_ACT_SILU || activation > ORACLE_ACT_RELU2)
    return ORACLE_ERR_ARG;
  const double* tab = decode_table(dtype);
  int bad = 0;
#pragma omp parallel for schedule(dynamic, 1) reduction(| : bad)
  for (int i = 0; i < n_tok; ++i) {
    int t = tok_list ? tok_list[i] : i;
    double* o = out + (int64_t)i * H;
    if (t < 0 || t >= T) {
      bad |= 1;
      continue;
    }
    int Fmax = F > S ? F : S;
    double* x = (double*)malloc(sizeof(double) * H);
    double* act = (double*)malloc(sizeof(double) * Fmax);
    double* y = (double*)malloc(sizeof(double) * H);
    double* u = act_noise ? (double*)malloc(sizeof(double) * Fmax) : NULL;
    double* nz = act_noise ? act_noise + (int64_t)i * H : NULL;
    for (int h = 0; h < H; ++h) x[h] = tab[hidden[(int64_t)t * H + h]];
    for (int h = 0; h < H; ++h) o[h] = 0.0;
    if (nz)
      for (int h = 0; h < H; ++h) nz[h] = 0.0;
    for (int j = 0; j < top_k; ++j) {
      int e = ids[(int64_t)t * top_k + j];
      if (e == -1) continue;
      if (e < -1 || e >= E) {
        bad |= 2;
        continue;
      }
      const uint16_t* wgu =
          expert_ptr(w_gate_up, expert_slot, e, gate_up_rows(activation, F) * H);
      const uint16_t* wd = expert_ptr(w_down, expert_slot, e, (int64_t)H * F);
      if (!wgu || !wd) {
        bad |= 1;
        continue;
      }
      double w = weights[(int64_t)t * top_k + j];
      act_rows(tab, wgu, x, H, F, activation, act);
      down_rows(tab, wd, act, H, F, y);
      for (int h = 0; h < H; ++h) o[h] += w * y[h];
      if (nz) down_noise(tab, wd, act, H, F, dtype, w * w, u, nz);
    }
    if (S > 0) {
      act_rows(tab, shared_w_gate_up, x, H, S, activation, act);
      down_rows(tab, shared_w_down, act, H, S, y);
      for (int h = 0; h < H; ++h) o[h] += y[h];
      if (nz) down_noise(tab, shared_w_down, act, H, S, dtype, 1.0, u, nz);
    }
    if (nz)
      for (int h = 0; h < H; ++h) nz[h] = sqrt(nz[h]);
    free(x);
    free(act);
    free(y);
    free(u);
  }
  if (bad & 2) return ORACLE_ERR_ID;
  if (bad) return ORACLE_ERR_ARG;
  return ORACLE_OK;
}

/*
 * Stage-level references used by the per-stage parity tests.
 *
 * oracle_expert_act: act[r, :] for n_rows input rows x_bits[r, :] (dtype bits, [n_rows, H]) all
 * routed to the expert given per row in expert_of_row[r] (-1: row left at 0).
 */
int oracle_expert_act(int n_rows, int H, int F, int dtype, int activation, const uint16_t* x_bits,
                      const int32_t* expert_of_row, const uint16_t* w_gate_up, double* act) {
  if (n_rows < 0 || H <= 0 || F <= 0 || activation < ORACLE_ACT_SILU ||
      activation > ORACLE_ACT_RELU2)
    return ORACLE_ERR_ARG;
  const double* tab = decode_table(dtype);
#pragma omp parallel for schedule(dynamic, 4)
  for (int r = 0; r < n_rows; ++r) {
    int e = expert_of_row[r];
    double* a = act + (int64_t)r * F;
    if (e < 0) {
      for (int f = 0; f < F; ++f) a[f] = 0.0;
      continue;
    }
    double* x = (double*)malloc(sizeof(double) * H);
    for (int h = 0; h < H; ++h) x[h] = tab[x_bits[(int64_t)r * H + h]];
    act_rows(tab, w_gate_up + (int64_t)e * gate_up_rows(activation, F) * H, x, H, F, activation,
             a);
    free(x);
  }
  return ORACLE_OK;
}

/* oracle_expert_down: y[r, :] = scale[r] * W_down[expert_of_row[r]] . act_bits[r, :]. */
int oracle_expert_down(int n_rows, int H, int F, int dtype, const uint16_t* act_bits,
                       const int32_t* expert_of_row, const double* scale,
                       const uint16_t* w_down, double* y) {
  if (n_rows < 0 || H <= 0 || F <= 0) return ORACLE_ERR_ARG;
  const double* tab = decode_table(dtype);
#pragma omp parallel for schedule(dynamic, 4)
  for (int r = 0; r < n_rows; ++r) {
    int e = expert_of_row[r];
    double* o = y + (int64_t)r * H;
    if (e < 0) {
      for (int h = 0; h < H; ++h) o[h] = 0.0;
      continue;
    }
    double* a = (double*)malloc(sizeof(double) * F);
    for (int f = 0; f < F; ++f) a[f] = tab[act_bits[(int64_t)r * F + f]];
    down_rows(tab, w_down + (int64_t)e * H * F, a, H, F, o);
    for (int h = 0; h < H; ++h) o[h] *= scale[r];
    free(a);
  }
  return ORACLE_OK;
}

/*
 * oracle_combine (TileOPs "MoE" page, op MoEPostPermuteFwd; aiter PR #5973 "Changes",
 * sorted_sum): out[t, :] = sum_j rows[inv_route[t*k+j], :] (+ shared[t, :]), skipping routes
 * whose inv_route is -1.  The route weight is already inside rows (it is applied by the down
 * projection stage), so this is a plain sum.
 */
int oracle_combine(int T, int H, int top_k, int dtype, const uint16_t* rows_bits,
                   const int32_t* inv_route, const uint16_t* shared_bits, double* out) {
  if (T < 0 || H <= 0 || top_k <= 0) return ORACLE_ERR_ARG;
  const double* tab = decode_table(dtype);
  for (int t = 0; t < T; ++t) {
    double* o = out + (int64_t)t * H;
    for (int h = 0; h < H; ++h) o[h] = shared_bits ? tab[shared_bits[(int64_t)t * H + h]] : 0.0;
    for (int j = 0; j < top_k; ++j) {
      int p = inv_route[(int64_t)t * top_k + j];
      if (p < 0) continue;
      for (int h = 0; h < H; ++h) o[h] += tab[rows_bits[(int64_t)p * H + h]];
    }
  }
  return ORACLE_OK;
}

/* ------------------------------------------------------------------------------------------ */
/* NVFP4 weights (flashinfer PR #4048 W4A16: NVFP4 weights decoded for a BF16 MMA, the FP32     */
/* per-expert scale applied to the FP32 accumulator; "W4A16 FP32 weight-scale placement          */
/* ablation").  A weight is  W[r,k] = e2m1(q) * e4m3(sf[r, k/16]) * alpha[expert]  with two     */
/* E2M1 codes per byte of q[r, k/2] (element 2i in the low nibble, 2i+1 in the high nibble) and  */
/* one E4M3 block scale per 16 consecutive k.  The two minifloats are decoded from their         */
/* definitions (OCP 8-bit and 4-bit floating point):                                           */
/*   E2M1: sign bit 3, exponent bits 2..1 (bias 1), mantissa bit 0, no inf/NaN;                 */
/*   E4M3: sign bit 7, exponent bits 6..3 (bias 7), mantissa bits 2..0, S.1111.111 is NaN,       */
/*         no inf.                                                                              */
/* ------------------------------------------------------------------------------------------ */

double oracle_e2m1_to_double(int code) {
  const int s = (code >> 3) & 1, e = (code >> 1) & 3, m = code & 1;
  const double mag = e == 0 ? 0.5 * m : ldexp(1.0 + 0.5 * m, e - 1);
  return s ? -mag : mag;
}

double oracle_e4m3_to_double(int bits) {
  const int s = (bits >> 7) & 1, e = (bits >> 3) & 15, m = bits & 7;
  double mag;
  if (e == 15 && m == 7)
    mag = NAN;
  else if (e == 0)
    mag = ldexp(m / 8.0, -6);
  else
    mag = ldexp(1.0 + m / 8.0, e - 7);
  return s ? -mag : mag;
}

static double g_e2m1[16];
static double g_e4m3[256];
static int g_fp_ready = 0;

static void fp_tables(void) {
  if (g_fp_ready) return;
#pragma omp critical(oracle_fp_tables)
  {
    if (!g_fp_ready) {
      for (int c = 0; c < 16; ++c) g_e2m1[c] = oracle_e2m1_to_double(c);
      for (int b = 0; b < 256; ++b) g_e4m3[b] = oracle_e4m3_to_double(b);
      g_fp_ready = 1;
    }
  }
}

/* One NVFP4 matrix row: q [K/2] bytes, sf [K/16] bytes. */
static double nvfp4_elem(const uint8_t* q, const uint8_t* sf, int k) {
  const uint8_t byte = q[k >> 1];
  const int code = (k & 1) ? (byte >> 4) : (byte & 15);
  return g_e2m1[code] * g_e4m3[sf[k >> 4]];
}

/* Dequantise n_rows rows of K: out[r,k] = W[r,k] with alpha[r / rows_per_alpha]. */
int oracle_nvfp4_dequant(int64_t n_rows, int K, const uint8_t* q, const uint8_t* sf,
                         const float* alpha, int64_t rows_per_alpha, double* out) {
  if (n_rows < 0 || K <= 0 || K % 16 != 0 || rows_per_alpha <= 0) return ORACLE_ERR_ARG;
  fp_tables();
  for (int64_t r = 0; r < n_rows; ++r) {
    const double a = (double)alpha[r / rows_per_alpha];
    for (int k = 0; k < K; ++k)
      out[r * K + k] = nvfp4_elem(q + r * (K / 2), sf + r * (K / 16), k) * a;
  }
  return ORACLE_OK;
}

/* NVFP4 expert of `rows` rows of length K: bytes of q and sf per expert. */
typedef struct {
  const uint8_t* q;
  const uint8_t* sf;
  double alpha;
  int K;
} w4_mat;

static w4_mat w4_expert(const uint8_t* q, const uint8_t* sf, const float* alpha, int e,
                        int64_t rows, int K) {
  w4_mat m;
  m.q = q + (int64_t)e * rows * (K / 2);
  m.sf = sf + (int64_t)e * rows * (K / 16);
  m.alpha = (double)alpha[e];
  m.K = K;
  return m;
}

/* sum_k W[row, k] x[k] for an NVFP4 matrix (alpha applied to the sum, which is exact math). */
static double w4_dot(const w4_mat* m, int64_t row, const double* x) {
  const uint8_t* q = m->q + row * (m->K / 2);
  const uint8_t* sf = m->sf + row * (m->K / 16);
  double s = 0.0;
  for (int k = 0; k < m->K; ++k) s += nvfp4_elem(q, sf, k) * x[k];
  return m->alpha * s;
}

/* sum_k (W[row, k] u[k])^2 for an NVFP4 matrix, W including alpha. */
static double w4_dot_sq(const w4_mat* m, int64_t row, const double* u) {
  const uint8_t* q = m->q + row * (m->K / 2);
  const uint8_t* sf = m->sf + row * (m->K / 16);
  double s = 0.0;
  for (int k = 0; k < m->K; ++k) {
    const double c = m->alpha * nvfp4_elem(q, sf, k) * u[k];
    s += c * c;
  }
  return s;
}

static void act_rows_w4(const w4_mat* wgu, const double* x, int F, int activation, double* act) {
  for (int f = 0; f < F; ++f) {
    const double g = w4_dot(wgu, f, x);
    if (activation == ORACLE_ACT_RELU2) {
      const double r = g > 0.0 ? g : 0.0;
      act[f] = r * r;
      continue;
    }
    const double u = w4_dot(wgu, (int64_t)F + f, x);
    act[f] = activation == ORACLE_ACT_GELU_TANH ? gelu_tanh(g) * u : g / (1.0 + exp(-g)) * u;
  }
}

/*
 * oracle_moe_tokens_w4: oracle_moe_tokens with NVFP4 routed experts (no shared expert):
 *   w1q [E, R1, H/2], w1sf [E, R1, H/16], w1a [E]   (R1 = 2F gated, F for ReLU2)
 *   w2q [E, H, F/2],  w2sf [E, H, F/16],  w2a [E]
 * The activations (hidden) are 16-bit of `dtype`; the weight of each term is the NVFP4 value
 * above.  act_noise (nullable): as in oracle_moe_tokens, for act rounded to the 16-bit type
 * act_dtype (0 bf16, 1 f16).
 */
int oracle_moe_tokens_w4(int n_tok, const int32_t* tok_list, int T, int H, int E, int F,
                         int top_k, int dtype, int act_dtype, int activation,
                         const uint16_t* hidden,
                         const int32_t* ids, const double* weights, const uint8_t* w1q,
                         const uint8_t* w1sf, const float* w1a, const uint8_t* w2q,
                         const uint8_t* w2sf, const float* w2a, double* out,
                         double* act_noise) {
  if (n_tok < 0 || H <= 0 || E <= 0 || F <= 0 || top_k <= 0 || (dtype != 0 && dtype != 1) ||
      (act_dtype != 0 && act_dtype != 1) || activation < ORACLE_ACT_SILU ||
      activation > ORACLE_ACT_RELU2 || H % 16 || F % 16)
    return ORACLE_ERR_ARG;
  const double* tab = decode_table(dtype);
  fp_tables();
  const int64_t R1 = gate_up_rows(activation, F);
  int bad = 0;
#pragma omp parallel for schedule(dynamic, 1) reduction(| : bad)
  for (int i = 0; i < n_tok; ++i) {
    int t = tok_list ? tok_list[i] : i;
    double* o = out + (int64_t)i * H;
    if (t < 0 || t >= T) {
      bad |= 1;
      continue;
    }
    double* x = (double*)malloc(sizeof(double) * H);
    double* act = (double*)malloc(sizeof(double) * F);
    double* u = act_noise ? (double*)malloc(sizeof(double) * F) : NULL;
    double* nz = act_noise ? act_noise + (int64_t)i * H : NULL;
    for (int h = 0; h < H; ++h) x[h] = tab[hidden[(int64_t)t * H + h]];
    for (int h = 0; h < H; ++h) o[h] = 0.0;
    if (nz)
      for (int h = 0; h < H; ++h) nz[h] = 0.0;
    for (int j = 0; j < top_k; ++j) {
      int e = ids[(int64_t)t * top_k + j];
      if (e == -1) continue;
      if (e < -1 || e >= E) {
        bad |= 2;
        continue;
      }
      const w4_mat m1 = w4_expert(w1q, w1sf, w1a, e, R1, H);
      const w4_mat m2 = w4_expert(w2q, w2sf, w2a, e, H, F);
      act_rows_w4(&m1, x, F, activation, act);
      const double w = weights[(int64_t)t * top_k + j];
      for (int h = 0; h < H; ++h) o[h] += w * w4_dot(&m2, h, act);
      if (nz) {
        for (int f = 0; f < F; ++f) u[f] = half_ulp16(act_dtype, act[f]);
        for (int h = 0; h < H; ++h) nz[h] += w * w * w4_dot_sq(&m2, h, u);
      }
    }
    if (nz)
      for (int h = 0; h < H; ++h) nz[h] = sqrt(nz[h]);
    free(x);
    free(act);
    free(u);
  }
  if (bad & 2) return ORACLE_ERR_ID;
  if (bad) return ORACLE_ERR_ARG;
  return ORACLE_OK;
}

/* Stage references with NVFP4 weights: act rows (gate/up) and route-scaled down rows. */
int oracle_expert_act_w4(int n_rows, int H, int F, int dtype, int activation,
                         const uint16_t* x_bits, const int32_t* expert_of_row, const uint8_t* w1q,
                         const uint8_t* w1sf, const float* w1a, double* act) {
  if (n_rows < 0 || H <= 0 || F <= 0 || H % 16 || activation < ORACLE_ACT_SILU ||
      activation > ORACLE_ACT_RELU2)
    return ORACLE_ERR_ARG;
  const double* tab = decode_table(dtype);
  fp_tables();
  const int64_t R1 = gate_up_rows(activation, F);
#pragma omp parallel for schedule(dynamic, 4)
  for (int r = 0; r < n_rows; ++r) {
    int e = expert_of_row[r];
    double* a = act + (int64_t)r * F;
    if (e < 0) {
      for (int f = 0; f < F; ++f) a[f] = 0.0;
      continue;
    }
    double* x = (double*)malloc(sizeof(double) * H);
    for (int h = 0; h < H; ++h) x[h] = tab[x_bits[(int64_t)r * H + h]];
    const w4_mat m1 = w4_expert(w1q, w1sf, w1a, e, R1, H);
    act_rows_w4(&m1, x, F, activation, a);
    free(x);
  }
  return ORACLE_OK;
}

int oracle_expert_down_w4(int n_rows, int H, int F, int dtype, const uint16_t* act_bits,
                          const int32_t* expert_of_row, const double* scale, const uint8_t* w2q,
                          const uint8_t* w2sf, const float* w2a, double* y) {
  if (n_rows < 0 || H <= 0 || F <= 0 || F % 16) return ORACLE_ERR_ARG;
  const double* tab = decode_table(dtype);
  fp_tables();
#pragma omp parallel for schedule(dynamic, 4)
  for (int r = 0; r < n_rows; ++r) {
    int e = expert_of_row[r];
    double* o = y + (int64_t)r * H;
    if (e < 0) {
      for (int h = 0; h < H; ++h) o[h] = 0.0;
      continue;
    }
    double* a = (double*)malloc(sizeof(double) * F);
    for (int f = 0; f < F; ++f) a[f] = tab[act_bits[(int64_t)r * F + f]];
    const w4_mat m2 = w4_expert(w2q, w2sf, w2a, e, H, F);
    for (int h = 0; h < H; ++h) o[h] = scale[r] * w4_dot(&m2, h, a);
    free(a);
  }
  return ORACLE_OK;
}

/* ------------------------------------------------------------------------------------------ */
/* Standalone grouped GEMM and post-permute (TileOPs "MoE" page, ops MoEGroupedGemmFwd and     */
/* MoEPostPermuteFwd).                                                                         */
/* ------------------------------------------------------------------------------------------ */

/*
 * oracle_grouped_gemm: out[r, n] = sum_k a[r, k] * b[e(r), n, k] for the rows r of each group e.
 *   masked layout (max_m > 0): a [E, max_m, K], out [E, max_m, N]; group e owns rows
 *     e*max_m .. e*max_m + meta[e] - 1 (meta = valid rows per group, clamped to [0, max_m]);
 *   contiguous layout (max_m == 0): a [P, K], out [P, N]; meta [E] are the inclusive prefix
 *     sums of the groups' row counts (group e owns rows meta[e-1] .. meta[e] - 1, meta[-1] = 0).
 * activation 0: plain product (b [E, N, K]); activation 1: silu_and_mul, b [E, 2N, K] with the
 * gate rows first, out = SiLU(a.b_gate) * (a.b_up).  Rows outside every group are left at 0.
 */
int oracle_grouped_gemm(int E, int N, int K, int max_m, int64_t rows, int dtype, int activation,
                        const uint16_t* a, const uint16_t* b, const int32_t* meta, double* out) {
  if (E <= 0 || N <= 0 || K <= 0 || max_m < 0 || rows < 0 || (dtype != 0 && dtype != 1) ||
      (activation != 0 && activation != 1))
    return ORACLE_ERR_ARG;
  const double* tab = decode_table(dtype);
  const int64_t nb = (int64_t)(activation ? 2 : 1) * N;
  for (int64_t i = 0; i < rows * N; ++i) out[i] = 0.0;
  int bad = 0;
  for (int e = 0; e < E; ++e) {
    int64_t r0, r1;
    if (max_m > 0) {
      int m = meta[e] < 0 ? 0 : (meta[e] > max_m ? max_m : meta[e]);
      r0 = (int64_t)e * max_m;
      r1 = r0 + m;
    } else {
      r0 = e == 0 ? 0 : meta[e - 1];
      r1 = meta[e];
    }
    if (r0 < 0 || r1 < r0 || r1 > rows) {
      bad = 1;
      continue;
    }
    const uint16_t* be = b + (int64_t)e * nb * K;
#pragma omp parallel for schedule(dynamic, 4)
    for (int64_t r = r0; r < r1; ++r) {
      const uint16_t* ar = a + r * K;
      for (int n = 0; n < N; ++n) {
        double g = 0.0;
        for (int k = 0; k < K; ++k) g += tab[ar[k]] * tab[be[(int64_t)n * K + k]];
        if (activation) {
          double u = 0.0;
          for (int k = 0; k < K; ++k) u += tab[ar[k]] * tab[be[(int64_t)(N + n) * K + k]];
          g = g / (1.0 + exp(-g)) * u;
        }
        out[r * N + n] = g;
      }
    }
  }
  return bad ? ORACLE_ERR_ARG : ORACLE_OK;
}

/*
 * oracle_post_permute (TileOPs "MoE" page, op MoEPostPermuteFwd):
 *   out[t, :] = sum_j weights[t, j] * rows[inv[t*k + j], :]   (routes with inv = -1 skipped)
 */
int oracle_post_permute(int T, int H, int top_k, int dtype, const uint16_t* rows_bits,
                        const double* weights, const int32_t* inv, double* out) {
  if (T < 0 || H <= 0 || top_k <= 0 || (dtype != 0 && dtype != 1)) return ORACLE_ERR_ARG;
  const double* tab = decode_table(dtype);
  for (int t = 0; t < T; ++t) {
    double* o = out + (int64_t)t * H;
    for (int h = 0; h < H; ++h) o[h] = 0.0;
    for (int j = 0; j < top_k; ++j) {
      const int p = inv[(int64_t)t * top_k + j];
      if (p < 0) continue;
      const double w = weights[(int64_t)t * top_k + j];
      for (int h = 0; h < H; ++h) o[h] += w * tab[rows_bits[(int64_t)p * H + h]];
    }
  }
  return ORACLE_OK;
}

/*
 * oracle_grouped_gemm_fp8 (TileOPs "MoE" page, op MoEGroupedGemmFP8Fwd): the grouped GEMM of
 * E4M3 operands with f32 block scales, masked (max_m > 0) or contiguous (max_m == 0) layout as
 * in oracle_grouped_gemm:
 *   out[r, n] = sum_kb a_scale[r, kb] * b_scale[e, n/128, kb]
 *                      * sum_{k in block kb} e4m3(a[r, k]) * e4m3(b[e, n, k])
 * with k blocks of 128; a [rows, K] and b [E, N, K] are E4M3 bytes, a_scale [rows, ceil(K/128)]
 * and b_scale [E, ceil(N/128), ceil(K/128)] f32.
 */
int oracle_grouped_gemm_fp8(int E, int N, int K, int max_m, int64_t rows, const uint8_t* a,
                            const float* a_scale, const uint8_t* b, const float* b_scale,
                            const int32_t* meta, double* out) {
  if (E <= 0 || N <= 0 || K <= 0 || max_m < 0 || rows < 0) return ORACLE_ERR_ARG;
  fp_tables();
  const int kbs = (K + 127) / 128, nbs = (N + 127) / 128;
  for (int64_t i = 0; i < rows * N; ++i) out[i] = 0.0;
  int bad = 0;
  for (int e = 0; e < E; ++e) {
    int64_t r0, r1;
    if (max_m > 0) {
      int m = meta[e] < 0 ? 0 : (meta[e] > max_m ? max_m : meta[e]);
      r0 = (int64_t)e * max_m;
      r1 = r0 + m;
    } else {
      r0 = e == 0 ? 0 : meta[e - 1];
      r1 = meta[e];
    }
    if (r0 < 0 || r1 < r0 || r1 > rows) {
      bad = 1;
      continue;
    }
#pragma omp parallel for schedule(dynamic, 4)
    for (int64_t r = r0; r < r1; ++r) {
      for (int n = 0; n < N; ++n) {
        const uint8_t* br = b + ((int64_t)e * N + n) * K;
        double acc = 0.0;
        for (int kb = 0; kb < kbs; ++kb) {
          double part = 0.0;
          for (int k = kb * 128; k < K && k < kb * 128 + 128; ++k)
            part += g_e4m3[a[r * K + k]] * g_e4m3[br[k]];
          acc += (double)a_scale[r * kbs + kb] *
                 (double)b_scale[((int64_t)e * nbs + n / 128) * kbs + kb] * part;
        }
        out[r * N + n] = acc;
      }
    }
  }
  return bad ? ORACLE_ERR_ARG : ORACLE_OK;
}

int oracle_num_threads(void) {
#ifdef _OPENMP
  extern int omp_get_max_threads(void);
  return omp_get_max_threads();
#else
  return 1;
#endif
}
