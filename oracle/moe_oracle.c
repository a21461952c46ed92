/*
 * CPU oracle for the routed-expert FFN layer. TEST INFRASTRUCTURE ONLY.
 *
 * A plain, slow, obviously correct statement of what the layer computes, in
 * fp64, written to be checked against the pages by eye. Only the tests, the
 * smoke check and the benchmark's CPU-baseline leg load it; the CUDA library
 * shares no code, header, table or helper with it.
 *
 * The layer (one MoE block of a large MoE language model):
 *   logits  l[t,e] = sum_i W_r[e,i] x[t,i] + b[e]
 *   top-k   the k largest logits of token t, largest first, ties to the lower e
 *   gates   g[t,j] = softmax over the k selected logits
 *   expert  h = SiLU(W_gate x) * (W_up x),   part = W_down h
 *   combine y[t] = sum_j g[t,j] part(t, j) + s_t shared(x_t)
 *           s_t = 1 (no gate row), or s_t = sigmoid(w_sg . x_t) with a gate row
 *
 * Sources (page title, section):
 *   "Neural Server" technical page, "How one token and one prompt are
 *     processed": the router and top-k kernels emit 4 expert ids and 4 weights
 *     per token; resident experts then run as MXFP4 GEMVs.
 *   "Neural Server" technical page, "What it runs on and what it runs": 128
 *     experts per layer, four active per token, hidden size 2880, and the
 *     13,219,200-byte MXFP4 expert.
 *   "NInfer" Qwen3.8-Flash-Next notes, MoE execution: (token, expert) pairs are
 *     grouped by expert; a fused gate/up kernel, then a down kernel; weighted
 *     expert outputs are summed; expert weights are renormalised per token.
 *   "Nebula", "Description": the router selects experts and assigns them
 *     normalised weights; gate/up/down expert tensors.
 *   "Running Qwen3.8-Flash-Next on a 32 GB Mac with Transformers",
 *     architecture: routed experts plus one shared expert per layer; its table
 *     of MoE blocks that carry a gate, a shared_expert and a
 *     shared_expert_gate (Qwen2-MoE, Qwen3-Next, Qwen3.5-MoE, Qwen3.8).
 *   "Nebula", the table of components held on the GPU: "shared expert gate",
 *     F32, 0.000458 GiB = 48 layers x 2,560 x 4 bytes, i.e. one fp32 row of
 *     the hidden size per layer (48 layers and hidden size 2,560 per the
 *     Transformers page's model line): one scalar gate per token.
 * None of the pages defines MXFP4's values; they follow the OCP Microscaling
 * Formats (MX) v1.0 specification: E2M1 elements, one E8M0 scale per 32
 * consecutive elements along the reduction axis, value = E2M1 * 2^(e - 127).
 *
 * Readings where the pages are silent:
 *   nibble order: the low nibble of byte i is element 2i, the high nibble 2i+1;
 *   gate/up: one [2F x d] matrix per expert, rows [0,F) gate, rows [F,2F) up;
 *   SiLU(z) = z / (1 + exp(-z)); no biases, no clamp;
 *   gates: softmax over the k selected logits (equal to the softmax over all
 *   E logits renormalised over the selected k);
 *   ties in top-k go to the lower expert index;
 *   the shared expert is added with weight 1; with a shared-expert gate row
 *   w_sg [d] its output is scaled by sigmoid(w_sg . x_t) (the pages name the
 *   tensor and its size, not the formula; the sigmoid of a one-row
 *   projection is the plainest reading of a per-token gate).
 *
 * Canonical expert-major weight layout (one contiguous byte range per expert):
 *   codes : expert j at j * (3 F d / 2): gate/up [2F][d/2], then down [d][F/2]
 *   scales: expert j at j * (3 F d / 32): gate/up [2F][d/32], then down [d][F/32]
 *   the shared expert (ffn S) follows expert E-1 in both arrays.
 */
#include <math.h>
#include <stddef.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define ORACLE_OK 0
#define ORACLE_EINVAL -1
#define ORACLE_ENAN_SCALE -2
#define ORACLE_ENOMEM -3

/* E2M1 (OCP MX v1.0): 1 sign bit, 2 exponent bits (bias 1), 1 mantissa bit. */
double oracle_e2m1(int code) {
  static const double magnitude[8] = {0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0};
  double v = magnitude[code & 7];
  return (code & 8) ? -v : v;
}

/* E8M0 scale (OCP MX v1.0): 2^(e - 127); the byte 0xFF encodes NaN. */
double oracle_e8m0(int e) {
  if (e == 255) return NAN;
  return ldexp(1.0, e - 127);
}

/* Exact value of a bf16 bit pattern. */
double oracle_bf16(uint16_t bits) {
  uint32_t u = (uint32_t)bits << 16;
  float f;
  memcpy(&f, &u, sizeof f);
  return (double)f;
}

/* Element (r, c) of an MXFP4 matrix whose rows hold K elements (K % 32 == 0). */
double oracle_mx_element(const uint8_t* codes, const uint8_t* scales, int K, int r, int c) {
  uint8_t byte = codes[(size_t)r * (size_t)(K / 2) + (size_t)(c / 2)];
  int code = (c & 1) ? (byte >> 4) : (byte & 0x0F);
  int e = scales[(size_t)r * (size_t)(K / 32) + (size_t)(c / 32)];
  return oracle_e2m1(code) * oracle_e8m0(e);
}

size_t oracle_expert_code_bytes(int d, int f) { return (size_t)3 * (size_t)f * (size_t)d / 2; }
size_t oracle_expert_scale_bytes(int d, int f) { return (size_t)3 * (size_t)f * (size_t)d / 32; }

/* Router logits of one token: l[e] = sum_i W_r[e,i] x[i] + b[e], fp64, index order. */
void oracle_logits_token(const uint16_t* x, int d, const float* w_router, const float* bias, int E,
                         double* logits) {
  for (int e = 0; e < E; ++e) {
    double acc = 0.0;
    for (int i = 0; i < d; ++i) acc += (double)w_router[(size_t)e * d + i] * oracle_bf16(x[i]);
    logits[e] = acc + (bias ? (double)bias[e] : 0.0);
  }
}

/* Shared-expert gate of one token: s = 1 / (1 + exp(-z)), z = sum_i w_sg[i] x[i]
 * in fp64, index order. */
double oracle_shared_gate_token(const uint16_t* x, int d, const float* w_sg) {
  double z = 0.0;
  for (int i = 0; i < d; ++i) z += (double)w_sg[i] * oracle_bf16(x[i]);
  return 1.0 / (1.0 + exp(-z));
}

/* Top-k of one token: repeatedly take the largest remaining logit, the lower
 * expert index winning an exact tie. Gates are the softmax of the selected
 * logits, shifted by the largest for range. */
void oracle_topk_token(const double* logits, int E, int k, int32_t* ids, double* gates) {
  char* taken = (char*)calloc((size_t)E, 1);
  for (int j = 0; j < k; ++j) {
    int best = -1;
    for (int e = 0; e < E; ++e) {
      if (taken[e]) continue;
      if (best < 0 || logits[e] > logits[best]) best = e; /* strict '>' keeps the lower index on ties */
    }
    taken[best] = 1;
    ids[j] = best;
  }
  free(taken);
  double top = logits[ids[0]];
  double denom = 0.0;
  for (int j = 0; j < k; ++j) denom += exp(logits[ids[j]] - top);
  for (int j = 0; j < k; ++j) gates[j] = exp(logits[ids[j]] - top) / denom;
}

/* Counting sort of the P = T*k (token, slot) pairs by expert, stable in p = t*k + j.
 * counts[e], offsets[0..E] (exclusive prefix sum), perm[row] = p, inv[p] = row. */
void oracle_bucket(const int32_t* ids, int P, int E, int32_t* counts, int32_t* offsets, int32_t* perm,
                   int32_t* inv) {
  for (int e = 0; e < E; ++e) counts[e] = 0;
  for (int p = 0; p < P; ++p) counts[ids[p]] += 1;
  offsets[0] = 0;
  for (int e = 0; e < E; ++e) offsets[e + 1] = offsets[e] + counts[e];
  int row = 0;
  for (int e = 0; e < E; ++e)
    for (int p = 0; p < P; ++p)
      if (ids[p] == e) {
        perm[row] = p;
        if (inv) inv[p] = row;
        ++row;
      }
}

static int scales_finite(const uint8_t* scales, size_t n) {
  for (size_t i = 0; i < n; ++i)
    if (scales[i] == 255) return 0;
  return 1;
}

/* One expert (ffn f) on one input vector x[d] (fp64):
 *   gate_i = sum_c Wgu[i][c] x[c],  up_i = sum_c Wgu[f + i][c] x[c]   (i < f)
 *   h_i = SiLU(gate_i) * up_i
 *   out_r = sum_i Wd[r][i] h_i                                         (r < d)
 * codes/scales point at the expert's own byte range. h may be NULL. */
int oracle_expert_ffn(const uint8_t* codes, const uint8_t* scales, int d, int f, const double* x, double* h,
                      double* out) {
  if (d <= 0 || f <= 0 || d % 32 || f % 32) return ORACLE_EINVAL;
  if (!scales_finite(scales, oracle_expert_scale_bytes(d, f))) return ORACLE_ENAN_SCALE;
  const uint8_t* gu_codes = codes;
  const uint8_t* gu_scales = scales;
  const uint8_t* dn_codes = codes + (size_t)2 * f * d / 2;
  const uint8_t* dn_scales = scales + (size_t)2 * f * d / 32;
  double* hv = (double*)malloc(sizeof(double) * (size_t)f);
  if (!hv) return ORACLE_ENOMEM;
  for (int i = 0; i < f; ++i) {
    double gate = 0.0, up = 0.0;
    for (int c = 0; c < d; ++c) {
      gate += oracle_mx_element(gu_codes, gu_scales, d, i, c) * x[c];
      up += oracle_mx_element(gu_codes, gu_scales, d, f + i, c) * x[c];
    }
    double silu = gate / (1.0 + exp(-gate));
    hv[i] = silu * up;
    if (h) h[i] = hv[i];
  }
  for (int r = 0; r < d; ++r) {
    double acc = 0.0;
    for (int i = 0; i < f; ++i) acc += oracle_mx_element(dn_codes, dn_scales, f, r, i) * hv[i];
    out[r] = acc;
  }
  free(hv);
  return ORACLE_OK;
}

/* Routing of all T tokens: logits [T][E], ids [T][k], gates [T][k], and the
 * bucketing of the T*k pairs (counts [E], offsets [E+1], perm [T*k], inv [T*k]).
 * Any output pointer except ids may be NULL. */
int oracle_route(const uint16_t* x, int T, int d, const float* w_router, const float* bias, int E, int k,
                 double* logits, int32_t* ids, double* gates, int32_t* counts, int32_t* offsets, int32_t* perm,
                 int32_t* inv) {
  if (T < 0 || d <= 0 || E <= 0 || k <= 0 || k > E || !ids) return ORACLE_EINVAL;
  double* l = (double*)malloc(sizeof(double) * (size_t)E);
  double* g = (double*)malloc(sizeof(double) * (size_t)k);
  if (!l || !g) { free(l); free(g); return ORACLE_ENOMEM; }
  for (int t = 0; t < T; ++t) {
    oracle_logits_token(x + (size_t)t * d, d, w_router, bias, E, l);
    if (logits) memcpy(logits + (size_t)t * E, l, sizeof(double) * (size_t)E);
    oracle_topk_token(l, E, k, ids + (size_t)t * k, g);
    if (gates) memcpy(gates + (size_t)t * k, g, sizeof(double) * (size_t)k);
  }
  free(l);
  free(g);
  if (counts && offsets && perm) {
    oracle_bucket(ids, T * k, E, counts, offsets, perm, inv);
  }
  return ORACLE_OK;
}

/* Layer output of the listed tokens (fp64, unrounded):
 *   y[n] = sum_j g[t,j] * expert(ids[t,j], x_t) + s_t * shared(x_t),   t = tokens[n]
 * summed in slot order j, the shared expert (when S > 0) last; s_t = 1 when
 * w_shared_gate is NULL, else oracle_shared_gate_token(x_t) (a gate row needs
 * a shared expert). h_out (may be NULL) receives h of every (n, j) as
 * [n_tokens][k][F]. */
int oracle_layer_tokens(int d, int F, int E, int k, int S, const uint16_t* x, const float* w_router,
                        const float* bias, const uint8_t* codes, const uint8_t* scales, const int32_t* tokens,
                        int n_tokens, double* y, double* h_out, int32_t* ids_out, double* gates_out,
                        const float* w_shared_gate) {
  if (d <= 0 || F <= 0 || E <= 0 || k <= 0 || k > E || S < 0 || d % 32 || F % 32 || S % 32) return ORACLE_EINVAL;
  if (w_shared_gate && S == 0) return ORACLE_EINVAL;
  size_t cb = oracle_expert_code_bytes(d, F), sb = oracle_expert_scale_bytes(d, F);
  double* l = (double*)malloc(sizeof(double) * (size_t)E);
  double* xv = (double*)malloc(sizeof(double) * (size_t)d);
  double* part = (double*)malloc(sizeof(double) * (size_t)d);
  int32_t* ids = (int32_t*)malloc(sizeof(int32_t) * (size_t)k);
  double* g = (double*)malloc(sizeof(double) * (size_t)k);
  int rc = ORACLE_OK;
  if (!l || !xv || !part || !ids || !g) { rc = ORACLE_ENOMEM; goto done; }
  for (int n = 0; n < n_tokens; ++n) {
    const uint16_t* xt = x + (size_t)tokens[n] * d;
    for (int i = 0; i < d; ++i) xv[i] = oracle_bf16(xt[i]);
    oracle_logits_token(xt, d, w_router, bias, E, l);
    oracle_topk_token(l, E, k, ids, g);
    if (ids_out) memcpy(ids_out + (size_t)n * k, ids, sizeof(int32_t) * (size_t)k);
    if (gates_out) memcpy(gates_out + (size_t)n * k, g, sizeof(double) * (size_t)k);
    double* yn = y + (size_t)n * d;
    for (int r = 0; r < d; ++r) yn[r] = 0.0;
    for (int j = 0; j < k; ++j) {
      double* hj = h_out ? h_out + ((size_t)n * k + j) * F : NULL;
      rc = oracle_expert_ffn(codes + (size_t)ids[j] * cb, scales + (size_t)ids[j] * sb, d, F, xv, hj, part);
      if (rc) goto done;
      for (int r = 0; r < d; ++r) yn[r] += g[j] * part[r];
    }
    if (S > 0) {
      rc = oracle_expert_ffn(codes + (size_t)E * cb, scales + (size_t)E * sb, d, S, xv, NULL, part);
      if (rc) goto done;
      const double st = w_shared_gate ? oracle_shared_gate_token(xt, d, w_shared_gate) : 1.0;
      for (int r = 0; r < d; ++r) yn[r] += st * part[r];
    }
  }
done:
  free(l); free(xv); free(part); free(ids); free(g);
  return rc;
}

/* One expert shard's part of the layer output (fp64, unrounded), for expert
 * parallelism (one GPU per contiguous range of experts): routing over all E
 * experts as in oracle_layer_tokens, but only the pairs whose expert is in
 * [e_begin, e_end) contribute, in slot order, and the shared expert (scaled
 * as in oracle_layer_tokens) only when with_shared is nonzero. The shards of a
 * partition of [0, E), one of them with the shared expert, add up to the
 * layer output. */
int oracle_layer_tokens_shard(int d, int F, int E, int k, int S, const uint16_t* x, const float* w_router,
                              const float* bias, const uint8_t* codes, const uint8_t* scales, const int32_t* tokens,
                              int n_tokens, int e_begin, int e_end, int with_shared, const float* w_shared_gate,
                              double* y) {
  if (d <= 0 || F <= 0 || E <= 0 || k <= 0 || k > E || S < 0 || d % 32 || F % 32 || S % 32) return ORACLE_EINVAL;
  if (e_begin < 0 || e_end > E || e_begin > e_end || (w_shared_gate && S == 0)) return ORACLE_EINVAL;
  size_t cb = oracle_expert_code_bytes(d, F), sb = oracle_expert_scale_bytes(d, F);
  double* l = (double*)malloc(sizeof(double) * (size_t)E);
  double* xv = (double*)malloc(sizeof(double) * (size_t)d);
  double* part = (double*)malloc(sizeof(double) * (size_t)d);
  int32_t* ids = (int32_t*)malloc(sizeof(int32_t) * (size_t)k);
  double* g = (double*)malloc(sizeof(double) * (size_t)k);
  int rc = ORACLE_OK;
  if (!l || !xv || !part || !ids || !g) { rc = ORACLE_ENOMEM; goto done; }
  for (int n = 0; n < n_tokens; ++n) {
    const uint16_t* xt = x + (size_t)tokens[n] * d;
    for (int i = 0; i < d; ++i) xv[i] = oracle_bf16(xt[i]);
    oracle_logits_token(xt, d, w_router, bias, E, l);
    oracle_topk_token(l, E, k, ids, g);
    double* yn = y + (size_t)n * d;
    for (int r = 0; r < d; ++r) yn[r] = 0.0;
    for (int j = 0; j < k; ++j) {
      if (ids[j] < e_begin || ids[j] >= e_end) continue;
      rc = oracle_expert_ffn(codes + (size_t)ids[j] * cb, scales + (size_t)ids[j] * sb, d, F, xv, NULL, part);
      if (rc) goto done;
      for (int r = 0; r < d; ++r) yn[r] += g[j] * part[r];
    }
    if (S > 0 && with_shared) {
      rc = oracle_expert_ffn(codes + (size_t)E * cb, scales + (size_t)E * sb, d, S, xv, NULL, part);
      if (rc) goto done;
      const double st = w_shared_gate ? oracle_shared_gate_token(xt, d, w_shared_gate) : 1.0;
      for (int r = 0; r < d; ++r) yn[r] += st * part[r];
    }
  }
done:
  free(l); free(xv); free(part); free(ids); free(g);
  return rc;
}

/* ---------------------------------------------------------------- affine group-64 experts
 *
 * A second expert weight format on the pages: "Running Qwen3.8-Flash-Next on a
 * 32 GB Mac with Transformers", the table of weights ("3-bit MLX affine, group
 * 64, 2.15 MB per expert") and its comparison bullets ("a 16-bit scale and
 * bias per 64 weights", about 3.5 bits per weight). Readings (the pages give
 * neither formula nor packing): an element is w = scale * q + bias with q the
 * unsigned `bits`-bit code of its group of 64 along the reduction axis;
 * scale and bias are bf16; a row's codes form one little-endian bit stream,
 * element c in bits [bits*c, bits*c + bits) of the row (K * bits / 8 bytes).
 * Per expert: gate/up [2f][d] then down [d][f], codes then scales then biases,
 * each matrix row-major. */

/* Code c of row r of a packed matrix (rows of K codes of `bits` bits). */
int oracle_affine_code(const uint8_t* packed, int K, int bits, int r, int c) {
  const uint8_t* row = packed + (size_t)r * (size_t)K * (size_t)bits / 8;
  int q = 0;
  for (int b = 0; b < bits; ++b) {
    long bit = (long)c * bits + b;
    q |= ((row[bit / 8] >> (bit % 8)) & 1) << b;
  }
  return q;
}

/* Element (r, c): scale * q + bias of the element's group of 64. */
double oracle_affine_element(const uint8_t* packed, const uint16_t* scales, const uint16_t* biases, int K, int bits,
                             int r, int c) {
  size_t g = (size_t)r * (size_t)(K / 64) + (size_t)(c / 64);
  return oracle_bf16(scales[g]) * (double)oracle_affine_code(packed, K, bits, r, c) + oracle_bf16(biases[g]);
}

/* Bytes of one affine expert: packed codes of the 3 f d weights, then a bf16
 * scale and a bf16 bias per 64 of them. */
size_t oracle_affine_expert_bytes(int d, int f, int bits) {
  size_t n = (size_t)3 * (size_t)f * (size_t)d;
  return n * (size_t)bits / 8 + (n / 64) * 2 * 2;
}

/* One affine expert (ffn f) on one input vector x[d] (fp64); `expert` points
 * at its oracle_affine_expert_bytes(d, f, bits) bytes. Same arithmetic as
 * oracle_expert_ffn, with affine elements. */
int oracle_expert_ffn_affine(const uint8_t* expert, int d, int f, int bits, const double* x, double* out) {
  if (d <= 0 || f <= 0 || d % 64 || f % 64 || bits < 1 || bits > 8) return ORACLE_EINVAL;
  const size_t n_gu = (size_t)2 * f * d, n_dn = (size_t)d * f;
  const uint8_t* gu_codes = expert;
  const uint8_t* dn_codes = gu_codes + n_gu * (size_t)bits / 8;
  const uint16_t* gu_scales = (const uint16_t*)(dn_codes + n_dn * (size_t)bits / 8);
  const uint16_t* dn_scales = gu_scales + n_gu / 64;
  const uint16_t* gu_biases = dn_scales + n_dn / 64;
  const uint16_t* dn_biases = gu_biases + n_gu / 64;
  double* hv = (double*)malloc(sizeof(double) * (size_t)f);
  if (!hv) return ORACLE_ENOMEM;
  for (int i = 0; i < f; ++i) {
    double gate = 0.0, up = 0.0;
    for (int c = 0; c < d; ++c) {
      gate += oracle_affine_element(gu_codes, gu_scales, gu_biases, d, bits, i, c) * x[c];
      up += oracle_affine_element(gu_codes, gu_scales, gu_biases, d, bits, f + i, c) * x[c];
    }
    hv[i] = gate / (1.0 + exp(-gate)) * up;
  }
  for (int r = 0; r < d; ++r) {
    double acc = 0.0;
    for (int i = 0; i < f; ++i) acc += oracle_affine_element(dn_codes, dn_scales, dn_biases, f, bits, r, i) * hv[i];
    out[r] = acc;
  }
  free(hv);
  return ORACLE_OK;
}

/* The layer of oracle_layer_tokens with affine group-64 experts: the same
 * routing, gate weighting and shared expert (optionally gated), each expert
 * (ffn F, the shared one ffn S) evaluated by oracle_expert_ffn_affine from
 * its oracle_affine_expert_bytes(d, f, bits) bytes, experts back to back in
 * `experts` (routed 0..E-1, then the shared one). y is fp64 and unrounded. */
int oracle_layer_tokens_affine(int d, int F, int E, int k, int S, int bits, const uint16_t* x, const float* w_router,
                               const float* bias, const uint8_t* experts, const int32_t* tokens, int n_tokens,
                               double* y, int32_t* ids_out, double* gates_out, const float* w_shared_gate) {
  if (d <= 0 || F <= 0 || E <= 0 || k <= 0 || k > E || S < 0 || d % 64 || F % 64 || S % 64 || bits < 1 || bits > 8)
    return ORACLE_EINVAL;
  if (w_shared_gate && S == 0) return ORACLE_EINVAL;
  size_t eb = oracle_affine_expert_bytes(d, F, bits);
  double* l = (double*)malloc(sizeof(double) * (size_t)E);
  double* xv = (double*)malloc(sizeof(double) * (size_t)d);
  double* part = (double*)malloc(sizeof(double) * (size_t)d);
  int32_t* ids = (int32_t*)malloc(sizeof(int32_t) * (size_t)k);
  double* g = (double*)malloc(sizeof(double) * (size_t)k);
  int rc = ORACLE_OK;
  if (!l || !xv || !part || !ids || !g) { rc = ORACLE_ENOMEM; goto done; }
  for (int n = 0; n < n_tokens; ++n) {
    const uint16_t* xt = x + (size_t)tokens[n] * d;
    for (int i = 0; i < d; ++i) xv[i] = oracle_bf16(xt[i]);
    oracle_logits_token(xt, d, w_router, bias, E, l);
    oracle_topk_token(l, E, k, ids, g);
    if (ids_out) memcpy(ids_out + (size_t)n * k, ids, sizeof(int32_t) * (size_t)k);
    if (gates_out) memcpy(gates_out + (size_t)n * k, g, sizeof(double) * (size_t)k);
    double* yn = y + (size_t)n * d;
    for (int r = 0; r < d; ++r) yn[r] = 0.0;
    for (int j = 0; j < k; ++j) {
      rc = oracle_expert_ffn_affine(experts + (size_t)ids[j] * eb, d, F, bits, xv, part);
      if (rc) goto done;
      for (int r = 0; r < d; ++r) yn[r] += g[j] * part[r];
    }
    if (S > 0) {
      rc = oracle_expert_ffn_affine(experts + (size_t)E * eb, d, S, bits, xv, part);
      if (rc) goto done;
      const double st = w_shared_gate ? oracle_shared_gate_token(xt, d, w_shared_gate) : 1.0;
      for (int r = 0; r < d; ++r) yn[r] += st * part[r];
    }
  }
done:
  free(l); free(xv); free(part); free(ids); free(g);
  return rc;
}
