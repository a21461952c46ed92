// sm_103a kernels of the routed-expert FFN layer.
//
// Forward = seven stream-ordered steps:
//   prep_x   per-token power-of-two scaling of x into f16 (exact for bf16 x)
//   router   l[t,e] = W_r[e] . x_t + b[e] in fp32, with an error bound
//   topk     candidates from the bounds, their logits as double-float (hi + lo)
//            sums, warp top-k with lower-index tie break, softmax gates
//   bucket   counting sort of the T*k pairs by expert, and the work list
//   gateup   grouped MXFP4 GEMM on tensor cores: h = SiLU(gate) * up (moe_gemm.cu)
//   down     grouped MXFP4 GEMM: part = W_down h (moe_gemm.cu)
//   combine  y_t = sum_j g[t,j] part(t,j) + shared_t, slot order, one rounding
//
// Where the pages describe the step (page title, section):
//   router/top-k: "Neural Server" technical page, "How one token and one prompt
//     are processed" (router and top-k write 4 ids and 4 weights per token).
//   grouping by expert, fused gate/up then down, per-token summation of a row
//     over all its experts in a fixed order: "NInfer" Qwen3.8-Flash-Next notes,
//     MoE execution bullets; fixed-order reductions: "Neural Server", "The CPU
//     kernel".
//
// Numerics. MXFP4 weights decode exactly to f16 (cvt.rn.f16x2.e2m1x2); the
// E8M0 scale of each 32-element block is applied in fp32 to that block's
// partial MMA sum. x (bf16) enters the MMA as f16 after multiplication by
// 2^sigma_t with max|x_t| * 2^sigma_t in [2^14, 2^15): exact except for
// elements below max|x_t| * 2^-28. h enters the down MMA as two f16 terms
// (hi + lo, about 22 significant bits) with a power-of-two scale per 16
// elements. All accumulation is fp32; all reductions run in a fixed order, so
// a token's output bits do not depend on timing.
#include <stdint.h>

#include "moe_device.cuh"
#include "moe_internal.h"

namespace moe {
namespace {

using namespace dev;


// ---------------------------------------------------------------- prep_x

__global__ void __launch_bounds__(256) prep_x_kernel(FwdParams p) {
  const int t = blockIdx.x;
  const uint16_t* xt = p.x + (size_t)t * p.d;
  __shared__ float wmax[8];
  float m = 0.f;
  for (int i = threadIdx.x; i < p.d; i += blockDim.x) m = fmaxf(m, fabsf(__uint_as_float((uint32_t)xt[i] << 16)));
  for (int o = 16; o; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
  if ((threadIdx.x & 31) == 0) wmax[threadIdx.x >> 5] = m;
  __syncthreads();
  m = 0.f;
  for (int w = 0; w < (int)(blockDim.x >> 5); ++w) m = fmaxf(m, wmax[w]);
  const int s = f16_headroom_exponent(m);
  const float sc = pow2f(s);
  __half* dst = reinterpret_cast<__half*>(p.x16) + (size_t)t * p.d64;
  for (int i = threadIdx.x; i < p.d; i += blockDim.x)
    dst[i] = __float2half_rn(__uint_as_float((uint32_t)xt[i] << 16) * sc);
  if (threadIdx.x == 0) p.xinv[t] = pow2f(-s);
}

// ---------------------------------------------------------------- router

// The router in two passes. Pass 1 (router_fp32_kernel): every logit in fp32
// by fused multiply-adds, 64 elements of d per partial sum, the partial sums
// added in order, then the bias: a sum in which every product passes at most
// D = 64 + ceil(d / 64) roundings, so |fp32 - exact| <= gamma_D sum|x_i w_i|
// + 2^-23 |logit| with gamma_D = D u / (1 - D u), u = 2^-24, and
// sum|x_i w_i| <= |x|_2 |w_e|_2 (Cauchy-Schwarz); the same pass bounds the
// two norms from above. Pass 2 (topk_kernel): per token, the k-th largest
// lower bound decides which experts can still be among the top k; only those
// get the double-float logit, and the top k, the order and the gates come from
// those values alone. The selection equals that of double-float logits for all
// experts: an expert whose upper bound is below the k-th largest lower bound
// is beaten by at least k others.
constexpr int kRfTok = 32, kRfExp = 32, kRfK = 64, kRfThreads = 128;

__device__ __forceinline__ float router_gamma(int d) {
  const float D = (float)(kRfK + (d + kRfK - 1) / kRfK);
  return D * 0x1p-24f / (1.f - D * 0x1p-24f);
}

// Block (32 tokens, 32 experts); thread (token pair tid / 8, expert quad tid % 8).
__global__ void __launch_bounds__(kRfThreads) router_fp32_kernel(FwdParams p) {
  __shared__ __align__(16) float xs[kRfK][kRfTok + 4];  // [k][token]
  __shared__ __align__(16) float ws[kRfK][kRfExp + 4];  // [k][expert]
  const int tid = threadIdx.x, t0 = blockIdx.x * kRfTok, e0 = blockIdx.y * kRfExp;
  const int tt = tid >> 3, te = tid & 7;
  float tot[2][4] = {};
  float xsq[2] = {0.f, 0.f}, wsq[4] = {0.f, 0.f, 0.f, 0.f};  // sums of squares of the rows this thread loads
  for (int kc = 0; kc < p.d; kc += kRfK) {
    for (int j = 0; j < 2; ++j) {  // x: 32 tokens x 64 elements, 8 per load
      const int r = tid + kRfThreads * j, tok = r >> 3, k8 = (r & 7) * 8;
      uint4 v = make_uint4(0u, 0u, 0u, 0u);
      if (t0 + tok < p.T && kc + k8 < p.d) v = __ldg(reinterpret_cast<const uint4*>(p.x + (size_t)(t0 + tok) * p.d + kc + k8));
      const uint32_t w4[4] = {v.x, v.y, v.z, v.w};
      float s = 0.f;
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        const float a = __uint_as_float(w4[q] << 16), b = __uint_as_float(w4[q] & 0xFFFF0000u);
        xs[k8 + 2 * q][tok] = a;
        xs[k8 + 2 * q + 1][tok] = b;
        s = fmaf(a, a, s);
        s = fmaf(b, b, s);
      }
      xsq[j] += s;
    }
    for (int j = 0; j < 4; ++j) {  // w: 32 experts x 64 elements, 4 per load
      const int r = tid + kRfThreads * j, ex = r >> 4, k4 = (r & 15) * 4;
      float4 v = make_float4(0.f, 0.f, 0.f, 0.f);
      if (e0 + ex < p.E && kc + k4 < p.d) v = __ldg(reinterpret_cast<const float4*>(p.w_router + (size_t)(e0 + ex) * p.d + kc + k4));
      ws[k4][ex] = v.x;
      ws[k4 + 1][ex] = v.y;
      ws[k4 + 2][ex] = v.z;
      ws[k4 + 3][ex] = v.w;
      wsq[j] += fmaf(v.x, v.x, fmaf(v.y, v.y, fmaf(v.z, v.z, v.w * v.w)));
    }
    __syncthreads();
    float c[2][4] = {};
#pragma unroll 16
    for (int k = 0; k < kRfK; ++k) {
      const float2 xv = *reinterpret_cast<const float2*>(&xs[k][2 * tt]);
      const float4 wv = *reinterpret_cast<const float4*>(&ws[k][4 * te]);
      const float xa[2] = {xv.x, xv.y}, wa[4] = {wv.x, wv.y, wv.z, wv.w};
#pragma unroll
      for (int a = 0; a < 2; ++a)
#pragma unroll
        for (int b = 0; b < 4; ++b) c[a][b] = fmaf(xa[a], wa[b], c[a][b]);
    }
#pragma unroll
    for (int a = 0; a < 2; ++a)
#pragma unroll
      for (int b = 0; b < 4; ++b) tot[a][b] += c[a][b];
    __syncthreads();
  }
#pragma unroll
  for (int a = 0; a < 2; ++a) {
    const int t = t0 + 2 * tt + a;
    if (t >= p.T) continue;
#pragma unroll
    for (int b = 0; b < 4; ++b) {
      const int e = e0 + 4 * te + b;
      if (e < p.E) p.logit_hi[(size_t)t * p.E + e] = p.bias ? tot[a][b] + p.bias[e] : tot[a][b];
    }
  }
  // norms, rounded up: the 8 (16) threads that loaded a token's (expert's) rows are adjacent lanes
  const float up = 1.f + (float)(p.d / 8 + 16) * 0x1p-22f;
  for (int j = 0; j < 2; ++j) {
    float s = xsq[j];
    for (int o = 1; o < 8; o <<= 1) s += __shfl_xor_sync(0xffffffffu, s, o);
    const int tok = (tid + kRfThreads * j) >> 3;
    if (blockIdx.y == 0 && (tid & 7) == 0 && t0 + tok < p.T) p.xnorm[t0 + tok] = sqrtf(s * up) * up;
  }
  for (int j = 0; j < 4; ++j) {
    float s = wsq[j];
    for (int o = 1; o < 16; o <<= 1) s += __shfl_xor_sync(0xffffffffu, s, o);
    const int ex = (tid + kRfThreads * j) >> 4;
    if (blockIdx.x == 0 && (tid & 15) == 0 && e0 + ex < p.E) p.wnorm[e0 + ex] = sqrtf(s * up) * up;
  }
}

// Double-float logit of expert e for token t by one warp (the value of lane 0,
// broadcast): lanes stride over d in groups of 8, then a fixed-shape tree.
__device__ __forceinline__ dd warp_logit_dd(const FwdParams& p, int t, int e) {
  const int lane = threadIdx.x & 31;
  dd acc{0.f, 0.f};
  const float* w = p.w_router + (size_t)e * p.d;
  const uint16_t* x = p.x + (size_t)t * p.d;
  for (int i8 = lane; i8 < p.d / 8; i8 += 32) {
    const uint4 xv = __ldg(reinterpret_cast<const uint4*>(x) + i8);
    const float4 w0 = __ldg(reinterpret_cast<const float4*>(w) + 2 * i8);
    const float4 w1 = __ldg(reinterpret_cast<const float4*>(w) + 2 * i8 + 1);
    const float wv[8] = {w0.x, w0.y, w0.z, w0.w, w1.x, w1.y, w1.z, w1.w};
    const uint32_t xw[4] = {xv.x, xv.y, xv.z, xv.w};
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      dd_mac(acc, __uint_as_float(xw[j] << 16), wv[2 * j]);
      dd_mac(acc, __uint_as_float(xw[j] & 0xFFFF0000u), wv[2 * j + 1]);
    }
  }
  for (int o = 16; o; o >>= 1) acc = dd_add(acc, dd_shfl_xor(acc, o));
  acc.hi = __shfl_sync(0xffffffffu, acc.hi, 0);
  acc.lo = __shfl_sync(0xffffffffu, acc.lo, 0);
  if (p.bias) acc = dd_add(acc, dd{p.bias[e], 0.f});
  return acc;
}

// ---------------------------------------------------------------- top-k and gates

constexpr int kTopkWarps = 8;
constexpr int kMaxEPerLane = 16;  // E <= 512

// One warp per token: the candidate set from the fp32 bounds, double-float
// logits of the candidates, then k rounds of a warp arg-max over them (value
// first, then the lower expert index) and the softmax of the k. The exported
// logits (hi + lo) are the double-float values for the candidates and the
// fp32 values (lo = 0) for the rest.
__global__ void __launch_bounds__(kTopkWarps * 32) topk_kernel(FwdParams p) {
  const int lane = threadIdx.x & 31;
  const int t = blockIdx.x * kTopkWarps + (threadIdx.x >> 5);
  if (t >= p.T) return;
  const int E = p.E, k = p.k;
  const float xb = router_gamma(p.d) * 1.01f * p.xnorm[t];
  float vh[kMaxEPerLane], vl[kMaxEPerLane], lb[kMaxEPerLane], ub[kMaxEPerLane];
#pragma unroll
  for (int i = 0; i < kMaxEPerLane; ++i) {
    const int e = lane + 32 * i;
    vh[i] = -INFINITY;
    vl[i] = 0.f;
    lb[i] = -INFINITY;
    ub[i] = -INFINITY;
    if (e < E) {
      const float l = p.logit_hi[(size_t)t * E + e];
      const float beta = fmaf(xb, p.wnorm[e], 0x1p-22f * fabsf(l)) + 0x1p-126f;
      vh[i] = l;
      lb[i] = l - beta;
      ub[i] = l + beta;
    }
  }
  // the k-th largest lower bound
  uint32_t taken = 0;
  float kth = -INFINITY;
  for (int j = 0; j < k; ++j) {
    float b = -INFINITY;
    int bi = 0x7fffffff;
#pragma unroll
    for (int i = 0; i < kMaxEPerLane; ++i)
      if (!((taken >> i) & 1u) && 32 * i + lane < E && (lb[i] > b || (lb[i] == b && 32 * i + lane < bi))) {
        b = lb[i];
        bi = 32 * i + lane;
      }
    for (int o = 16; o; o >>= 1) {
      const float ob = __shfl_xor_sync(0xffffffffu, b, o);
      const int oi = __shfl_xor_sync(0xffffffffu, bi, o);
      if (ob > b || (ob == b && oi < bi)) {
        b = ob;
        bi = oi;
      }
    }
    if ((bi & 31) == lane) taken |= 1u << (bi >> 5);
    kth = b;
  }
  // candidates: double-float logits
  uint32_t cand = 0;
#pragma unroll
  for (int i = 0; i < kMaxEPerLane; ++i) {
    const bool c = 32 * i + lane < E && ub[i] >= kth;
    if (c) cand |= 1u << i;
    unsigned cm = __ballot_sync(0xffffffffu, c);
    while (cm) {
      const int l = __ffs(cm) - 1;
      cm &= cm - 1;
      const dd v = warp_logit_dd(p, t, l + 32 * i);
      if (lane == l) {
        vh[i] = v.hi;
        vl[i] = v.lo;
      }
    }
  }
  for (int i = 0; i < kMaxEPerLane; ++i) {  // the exported logits
    const int e = lane + 32 * i;
    if (e < E) {
      p.logit_hi[(size_t)t * E + e] = vh[i];
      p.logit_lo[(size_t)t * E + e] = vl[i];
    }
  }
  taken = ~cand;
  float sel_h = 0.f, sel_l = 0.f, top_h = 0.f, top_l = 0.f;
  int sel_id = 0;
  for (int j = 0; j < k; ++j) {
    float bh = -INFINITY, bl = 0.f;
    int bi = 0x7fffffff;
#pragma unroll
    for (int i = 0; i < kMaxEPerLane; ++i) {
      if (!((taken >> i) & 1u) && dd_greater(vh[i], vl[i], lane + 32 * i, bh, bl, bi)) {
        bh = vh[i];
        bl = vl[i];
        bi = lane + 32 * i;
      }
    }
    for (int o = 16; o; o >>= 1) {
      const float oh = __shfl_xor_sync(0xffffffffu, bh, o);
      const float ol = __shfl_xor_sync(0xffffffffu, bl, o);
      const int oi = __shfl_xor_sync(0xffffffffu, bi, o);
      if (dd_greater(oh, ol, oi, bh, bl, bi)) {
        bh = oh;
        bl = ol;
        bi = oi;
      }
    }
    if ((bi & 31) == lane) taken |= 1u << (bi >> 5);
    if (j == 0) {
      top_h = bh;
      top_l = bl;
    }
    if (lane == j) {
      sel_h = bh;
      sel_l = bl;
      sel_id = bi;
    }
  }
  float ex = 0.f;
  if (lane < k) ex = expf((sel_h - top_h) + (sel_l - top_l));
  float sum = ex;
  for (int o = 16; o; o >>= 1) sum += __shfl_xor_sync(0xffffffffu, sum, o);
  if (lane < k) {
    p.ids[(size_t)t * k + lane] = sel_id;
    p.gates[(size_t)t * k + lane] = ex / sum;
  }
}

// ---------------------------------------------------------------- bucketing and work list

constexpr int kBucketThreads = 1024;

// Counting sort of the P = T*k pairs by expert (histogram, exclusive scan,
// ranks within a bucket in pair order), then one work-list slot per expert
// that received pairs (expert order) and the shared expert last.
__global__ void __launch_bounds__(kBucketThreads) bucket_kernel(FwdParams p) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int E = p.E, T = p.T, P = p.P;
  __shared__ int cnt[512];
  __shared__ int run[512];
  __shared__ int offs[513];
  for (int e = threadIdx.x; e < E; e += kBucketThreads) {
    cnt[e] = 0;
    run[e] = 0;
  }
  __syncthreads();
  for (int q = threadIdx.x; q < P; q += kBucketThreads) atomicAdd(&cnt[p.ids[q]], 1);
  __syncthreads();
  if (threadIdx.x == 0) {
    int acc = 0;
    for (int e = 0; e < E; ++e) {
      offs[e] = acc;
      acc += cnt[e];
    }
    offs[E] = acc;
  }
  __syncthreads();
  for (int e = threadIdx.x; e <= E; e += kBucketThreads) {
    p.offsets[e] = offs[e];
    if (e < E) p.counts[e] = cnt[e];
  }
  if (warp == 0) {
    for (int base = 0; base < P; base += 32) {
      const int q = base + lane;
      const bool valid = q < P;
      const int e = valid ? p.ids[q] : -1 - lane;
      const unsigned same = __match_any_sync(0xffffffffu, e);
      const int rank = __popc(same & ((1u << lane) - 1u));
      const int before = valid ? run[e] : 0;
      __syncwarp();
      if (valid && rank == 0) run[e] = before + __popc(same);
      __syncwarp();
      if (valid) {
        const int pos = offs[e] + before + rank;
        p.perm[pos] = q;
        p.inv[q] = pos;
      }
    }
  }
  if (threadIdx.x == 32) {
    int ns = 0, gu = 0, dn = 0, pn = 0;
    for (int e = 0; e < E; ++e) {
      if (cnt[e] == 0) continue;
      p.slot_expert[ns] = e;
      p.slot_q0[ns] = offs[e];
      p.slot_n[ns] = cnt[e];
      p.gu_prefix[ns] = gu;
      p.dn_prefix[ns] = dn;
      if (p.tc_gateup) p.panel_prefix[ns] = pn;
      pn += (cnt[e] + kTcGemmRows - 1) / kTcGemmRows;
      const int blocks = (cnt[e] + kGemmRows - 1) / kGemmRows;
      gu += p.tc_gateup ? (cnt[e] + kTcGemmRows - 1) / kTcGemmRows * ((p.F / 16 + 3) / 4)
                        : blocks * ((p.F / 16 + kGemmTiles - 1) / kGemmTiles);
      dn += p.tc_gateup ? (cnt[e] + kTcGemmRows - 1) / kTcGemmRows * tc_dtiles(p.d)
                        : blocks * ((p.d / 16 + kGemmTiles - 1) / kGemmTiles);
      ++ns;
    }
    if (p.S > 0 && T > 0) {
      p.slot_expert[ns] = E;
      p.slot_q0[ns] = P;
      p.slot_n[ns] = T;
      p.gu_prefix[ns] = gu;
      p.dn_prefix[ns] = dn;
      if (p.tc_gateup) p.panel_prefix[ns] = pn;
      pn += (T + kTcGemmRows - 1) / kTcGemmRows;
      const int blocks = (T + kGemmRows - 1) / kGemmRows;
      gu += p.tc_gateup ? (T + kTcGemmRows - 1) / kTcGemmRows * ((p.S / 16 + 3) / 4)
                        : blocks * ((p.S / 16 + kGemmTiles - 1) / kGemmTiles);
      dn += p.tc_gateup ? (T + kTcGemmRows - 1) / kTcGemmRows * tc_dtiles(p.d)
                        : blocks * ((p.d / 16 + kGemmTiles - 1) / kGemmTiles);
      ++ns;
    }
    p.gu_prefix[ns] = gu;
    p.dn_prefix[ns] = dn;
    if (p.tc_gateup) p.panel_prefix[ns] = pn;
    *p.n_slots = ns;
  }
}

// ---------------------------------------------------------------- combine

__global__ void __launch_bounds__(256) combine_kernel(FwdParams p) {
  const int t = blockIdx.y;
  const int r = blockIdx.x * blockDim.x + threadIdx.x;
  if (r >= p.d) return;
  float acc = 0.f;
  for (int j = 0; j < p.k; ++j) {
    const int pj = t * p.k + j;
    acc = fmaf(p.gates[pj], p.part[(size_t)p.inv[pj] * p.d + r], acc);
  }
  if (p.S > 0) acc += p.part[(size_t)(p.P + t) * p.d + r];
  if (p.out_f32) reinterpret_cast<float*>(p.out)[(size_t)t * p.d + r] = acc;
  else reinterpret_cast<__nv_bfloat16*>(p.out)[(size_t)t * p.d + r] = __float2bfloat16_rn(acc);
}

// ---------------------------------------------------------------- repack

__device__ __forceinline__ int gu_row(int tau, int r) { return 32 * (tau >> 1) + 8 * (r >> 2) + 4 * (tau & 1) + (r & 3); }

// One thread per (expert, tile, lane). Canonical matrix: codes [R][K/2], scales [R][K/32].
__global__ void repack_kernel(const uint8_t* codes, const uint8_t* scales, int n_exp, int d, int f,
                              size_t canon_code_stride, size_t canon_scale_stride, uint8_t* out, size_t out_stride,
                              int* err) {
  const int K64d = k64_tiles(d), K64f = k64_tiles(f);
  const long long gu_tiles = (long long)(f / 16) * K64d * 2;
  const long long dn_tiles = (long long)(d / 16) * K64f;
  const long long per_exp = gu_tiles + dn_tiles;
  const long long total = per_exp * n_exp * 32;
  for (long long gid = (long long)blockIdx.x * blockDim.x + threadIdx.x; gid < total;
       gid += (long long)gridDim.x * blockDim.x) {
    const int lane = (int)(gid & 31);
    const long long tile = gid >> 5;
    const int x = (int)(tile / per_exp);
    const long long tl = tile % per_exp;
    const int g = lane >> 2, c = lane & 3;
    const uint8_t* mc;
    const uint8_t* ms;
    int K, kt, rows[2];
    uint8_t* dst = out + (size_t)x * out_stride + (size_t)tl * kTileBytes;
    if (tl < gu_tiles) {
      const int tau = (int)(tl / (2 * K64d));
      const int rem = (int)(tl % (2 * K64d));
      kt = rem >> 1;
      const int half = rem & 1;
      K = d;
      mc = codes + (size_t)x * canon_code_stride;
      ms = scales + (size_t)x * canon_scale_stride;
      rows[0] = half * f + gu_row(tau, g);
      rows[1] = half * f + gu_row(tau, g + 8);
    } else {
      const long long t2 = tl - gu_tiles;
      const int mt = (int)(t2 / K64f);
      kt = (int)(t2 % K64f);
      K = f;
      mc = codes + (size_t)x * canon_code_stride + (size_t)f * d;
      ms = scales + (size_t)x * canon_scale_stride + (size_t)2 * f * d / 32;
      rows[0] = 16 * mt + g;
      rows[1] = 16 * mt + g + 8;
    }
    __align__(16) uint8_t cb[16];
    __align__(4) uint8_t sb[4];
#pragma unroll
    for (int bb = 0; bb < 2; ++bb) {
      const int blk = 2 * kt + bb;
#pragma unroll
      for (int rr = 0; rr < 2; ++rr) {
        const bool in = blk < K / 32;
#pragma unroll
        for (int i = 0; i < 4; ++i)
          cb[8 * bb + 4 * rr + i] = in ? mc[(size_t)rows[rr] * (K / 2) + blk * 16 + 4 * c + i] : (uint8_t)0;
        const uint8_t s = in ? ms[(size_t)rows[rr] * (K / 32) + blk] : (uint8_t)127;
        if (s == 255) atomicExch(err, 1);
        sb[2 * bb + rr] = s;
      }
    }
    *reinterpret_cast<uint4*>(dst + 16 * lane) = *reinterpret_cast<const uint4*>(cb);
    if (c == 0) *reinterpret_cast<uint32_t*>(dst + kTileCodeBytes + 4 * g) = *reinterpret_cast<const uint32_t*>(sb);
  }
}

}  // namespace

const char* const kForwardPhaseNames = "route,gateup,down,combine";

cudaError_t launch_forward(const FwdParams& p, cudaStream_t stream, int num_sms, cudaEvent_t const* events) {
  if (p.T == 0) return cudaSuccess;
  if (events) cudaEventRecord(events[0], stream);
  prep_x_kernel<<<p.T, 256, 0, stream>>>(p);
  router_fp32_kernel<<<dim3((p.T + kRfTok - 1) / kRfTok, (p.E + kRfExp - 1) / kRfExp), kRfThreads, 0, stream>>>(p);
  topk_kernel<<<(p.T + kTopkWarps - 1) / kTopkWarps, kTopkWarps * 32, 0, stream>>>(p);
  bucket_kernel<<<1, kBucketThreads, 0, stream>>>(p);
  if (events) cudaEventRecord(events[1], stream);
  cudaError_t e = p.tc_gateup ? launch_gemm_gateup_tc(p, stream, num_sms) : launch_gemm_gateup(p, stream, num_sms);
  if (e != cudaSuccess) return e;
  if (events) cudaEventRecord(events[2], stream);
  e = p.tc_gateup ? launch_gemm_down_tc(p, stream, num_sms) : launch_gemm_down(p, stream, num_sms);
  if (e != cudaSuccess) return e;
  if (events) cudaEventRecord(events[3], stream);
  combine_kernel<<<dim3((p.d + 255) / 256, p.T), 256, 0, stream>>>(p);
  if (events) cudaEventRecord(events[4], stream);
  return cudaGetLastError();
}

cudaError_t launch_route(const FwdParams& p, cudaStream_t stream) {
  if (p.T == 0) return cudaSuccess;
  router_fp32_kernel<<<dim3((p.T + kRfTok - 1) / kRfTok, (p.E + kRfExp - 1) / kRfExp), kRfThreads, 0, stream>>>(p);
  topk_kernel<<<(p.T + kTopkWarps - 1) / kTopkWarps, kTopkWarps * 32, 0, stream>>>(p);
  bucket_kernel<<<1, kBucketThreads, 0, stream>>>(p);
  return cudaGetLastError();
}

cudaError_t launch_repack(const uint8_t* codes, const uint8_t* scales, int n_exp, int d, int f,
                          size_t canon_code_stride, size_t canon_scale_stride, uint8_t* out, size_t out_stride,
                          int* err_flag, cudaStream_t stream) {
  repack_kernel<<<1024, 256, 0, stream>>>(codes, scales, n_exp, d, f, canon_code_stride, canon_scale_stride, out,
                                          out_stride, err_flag);
  return cudaGetLastError();
}

}  // namespace moe
