// sm_103a kernels of the routed-expert FFN layer.
//
// Forward = seven stream-ordered steps:
//   prep_x   per-token power-of-two scaling of x into f16 (exact for bf16 x)
//   router   l[t,e] = W_r[e] . x_t + b[e] in fp32, with an error bound
//   topk     candidates from the bounds, their logits as double-float (hi + lo)
//            sums, warp top-k with lower-index tie break, softmax gates
//            (T <= kRouteDDMaxT: every logit as a double-float sum over all SMs
//            instead, and the top-k at the start of the bucketing kernel)
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

// f16 x of token t (x * 2^sigma_t), 2^-sigma_t and, for affine experts, the
// group sums: by one block of 256 threads (all of them call it).
__device__ void prep_x_token(const FwdParams& p, int t) {
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
  if (p.xgsum) {  // affine experts: the sum of every 64-element group of the f16 x, one warp per group
    __syncthreads();  // (fixed order: element pairs per lane, then a butterfly over the lanes)
    const int lane = threadIdx.x & 31;
    for (int g = threadIdx.x >> 5; g < p.d / 64; g += blockDim.x >> 5) {
      float a = __half2float(dst[64 * g + 2 * lane]) + __half2float(dst[64 * g + 2 * lane + 1]);
      for (int o = 1; o < 32; o <<= 1) a += __shfl_xor_sync(0xffffffffu, a, o);
      if (lane == 0) p.xgsum[(size_t)t * p.xg_pitch + g] = a * 0x1p-24f;  // the scale of the codes' f16 form
    }
  }
}

__global__ void __launch_bounds__(256) prep_x_kernel(FwdParams p) {
  pdl_enter();
  prep_x_token(p, blockIdx.x);
}

// ---------------------------------------------------------------- router

// The router in two passes. Pass 1 (router_fp32_kernel): every logit in fp32
// by fused multiply-adds, 128 elements of d per partial sum, the partial sums
// added in order within each of rsplit ranges of d (one per block column), the
// ranges added in order and then the bias by the top-k kernel: a sum in which
// every product passes at most D = 128 + ceil(d / 128) + 3 roundings, so
// |fp32 - exact| <= gamma_D sum|x_i w_i| + 2^-23 |logit| with
// gamma_D = D u / (1 - D u), u = 2^-24, and sum|x_i w_i| <= |x|_2 |w_e|_2
// (Cauchy-Schwarz); the same pass sums the squares for the two norms. Pass 2
// (topk_kernel): per token, the k-th largest lower bound decides which experts
// can still be among the top k; only those get the double-float logit, and
// the top k, the order and the gates come from those values alone. The
// selection equals that of double-float logits for all experts: an expert
// whose upper bound is below the k-th largest lower bound is beaten by at
// least k others.
constexpr int kRfTok = 64, kRfExp = 32, kRfK = 128, kRfThreads = 128;
constexpr int kRfKS = 64;  // elements of d staged in shared memory at a time (half a partial sum)

__device__ __forceinline__ float router_gamma(int d) {
  const float D = (float)(kRfK + (d + kRfK - 1) / kRfK + 3);
  return D * 0x1p-24f / (1.f - D * 0x1p-24f);
}

// Block (64 tokens, 32 experts, range z of d); thread (token quad tid / 8,
// expert quad tid % 8) keeps 16 products in registers, two 16-byte shared
// loads per 16 multiply-adds. Each partial sum runs over 128 elements of d
// (two staged halves of 64) from zero, then is added to the thread's total.
// Loads: x rows as 8-element groups (thread t takes token t % 64), W_r rows as
// 4-element groups (thread t takes expert t % 32); warps step through K, so
// the transposed stores to shared memory hit 32 banks. The next half is
// loaded into registers while the current one is multiplied out of shared
// memory. The squares of the loaded x (W_r) elements are summed by the 2 (4)
// threads of a token (an expert) and added in thread order at the end.
__global__ void __launch_bounds__(kRfThreads) router_fp32_kernel(FwdParams p) {
  pdl_enter();
  __shared__ __align__(16) float xs[kRfKS][kRfTok];  // [k][token]
  __shared__ __align__(16) float ws[kRfKS][kRfExp];  // [k][expert]
  __shared__ float nsq[kRfThreads];
  constexpr int kXL = kRfTok * kRfKS / 8 / kRfThreads;  // 8-element x loads per thread and half
  constexpr int kWL = kRfExp * kRfKS / 4 / kRfThreads;  // 4-element W_r loads per thread and half
  const int tid = threadIdx.x;
  const int t0 = blockIdx.x * kRfTok, e0 = blockIdx.y * kRfExp, z = blockIdx.z;
  const int nch = (p.d + kRfK - 1) / kRfK, cps = (nch + p.rsplit - 1) / p.rsplit;
  const int kbeg = z * cps * kRfK, kend = min(p.d, (z + 1) * cps * kRfK);
  const int tt = tid >> 3, te = tid & 7;
  const int xt = tid % kRfTok, xg = tid / kRfTok;  // load role: token row, first 8-element group
  const int we = tid % kRfExp, wg = tid / kRfExp;  // load role: expert row, first 4-element group
  float tot[4][4] = {}, c[4][4] = {};
  float xsq = 0.f, wsq = 0.f;
  uint4 xr[kXL];
  float4 wr[kWL];
  const bool xok = t0 + xt < p.T, wok = e0 + we < p.E;
  const uint16_t* xrow = p.x + (size_t)(t0 + xt) * p.d;
  const float* wrow = p.w_router + (size_t)(e0 + we) * p.d;
  auto load = [&](int kc) {
#pragma unroll
    for (int j = 0; j < kXL; ++j) {
      const int k8 = 8 * (xg + (kRfThreads / kRfTok) * j);
      xr[j] = make_uint4(0u, 0u, 0u, 0u);
      if (xok && kc + k8 < kend) xr[j] = __ldg(reinterpret_cast<const uint4*>(xrow + kc + k8));
    }
#pragma unroll
    for (int j = 0; j < kWL; ++j) {
      const int k4 = 4 * (wg + (kRfThreads / kRfExp) * j);
      wr[j] = make_float4(0.f, 0.f, 0.f, 0.f);
      if (wok && kc + k4 < kend) wr[j] = __ldg(reinterpret_cast<const float4*>(wrow + kc + k4));
    }
  };
  if (kbeg < kend) load(kbeg);
  for (int kc = kbeg; kc < kend; kc += kRfKS) {
#pragma unroll
    for (int j = 0; j < kXL; ++j) {
      const int k8 = 8 * (xg + (kRfThreads / kRfTok) * j);
      const uint32_t w4[4] = {xr[j].x, xr[j].y, xr[j].z, xr[j].w};
      float sq = 0.f;
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        const float a = __uint_as_float(w4[q] << 16), b = __uint_as_float(w4[q] & 0xFFFF0000u);
        xs[k8 + 2 * q][xt] = a;
        xs[k8 + 2 * q + 1][xt] = b;
        sq = fmaf(a, a, sq);
        sq = fmaf(b, b, sq);
      }
      xsq += sq;
    }
#pragma unroll
    for (int j = 0; j < kWL; ++j) {
      const int k4 = 4 * (wg + (kRfThreads / kRfExp) * j);
      ws[k4][we] = wr[j].x;
      ws[k4 + 1][we] = wr[j].y;
      ws[k4 + 2][we] = wr[j].z;
      ws[k4 + 3][we] = wr[j].w;
      wsq += fmaf(wr[j].x, wr[j].x, fmaf(wr[j].y, wr[j].y, fmaf(wr[j].z, wr[j].z, wr[j].w * wr[j].w)));
    }
    __syncthreads();
    if (kc + kRfKS < kend) load(kc + kRfKS);
#pragma unroll 16
    for (int k = 0; k < kRfKS; ++k) {
      const float4 xv = *reinterpret_cast<const float4*>(&xs[k][4 * tt]);
      const float4 wv = *reinterpret_cast<const float4*>(&ws[k][4 * te]);
      const float xa[4] = {xv.x, xv.y, xv.z, xv.w}, wa[4] = {wv.x, wv.y, wv.z, wv.w};
#pragma unroll
      for (int a = 0; a < 4; ++a)
#pragma unroll
        for (int b = 0; b < 4; ++b) c[a][b] = fmaf(xa[a], wa[b], c[a][b]);
    }
    // a partial sum ends every 128 elements of d (and at the end of the range)
    if (((kc - kbeg) / kRfKS) % (kRfK / kRfKS) == kRfK / kRfKS - 1 || kc + kRfKS >= kend) {
#pragma unroll
      for (int a = 0; a < 4; ++a)
#pragma unroll
        for (int b = 0; b < 4; ++b) {
          tot[a][b] += c[a][b];
          c[a][b] = 0.f;
        }
    }
    __syncthreads();
  }
  float* plane = p.logit_hi + (size_t)z * p.lstride;  // partial sums of range z
#pragma unroll
  for (int a = 0; a < 4; ++a) {
    const int t = t0 + 4 * tt + a;
    if (t >= p.T) continue;
#pragma unroll
    for (int b = 0; b < 4; ++b) {
      const int e = e0 + 4 * te + b;
      if (e < p.E) plane[(size_t)t * p.E + e] = tot[a][b];
    }
  }
  // sums of squares of range z: a token's (expert's) threads in thread order
  nsq[tid] = xsq;
  __syncthreads();
  if (tid < kRfTok && blockIdx.y == 0 && xok) {
    float sq = 0.f;
    for (int i = 0; i < kRfThreads / kRfTok; ++i) sq += nsq[tid + kRfTok * i];
    p.xsq[(size_t)z * p.lstride / p.E + t0 + tid] = sq;
  }
  __syncthreads();
  nsq[tid] = wsq;
  __syncthreads();
  if (tid < kRfExp && blockIdx.x == 0 && wok) {
    float sq = 0.f;
    for (int i = 0; i < kRfThreads / kRfExp; ++i) sq += nsq[tid + kRfExp * i];
    p.wsq[z * p.E + e0 + tid] = sq;
  }
}

// ---------------------------------------------------------------- top-k and gates

constexpr int kTopkThreads = 128;
constexpr int kTopkMaxE = 512;

// Double-float partial logits, over elements [k0, k1) of d, of up to 4
// experts es[0 .. n) for token t by one warp (the values of lane 0,
// broadcast): lanes stride over the range in groups of 8, one accumulator per
// expert, then a fixed-shape tree per expert.
__device__ __forceinline__ void warp_logits_dd(const FwdParams& p, int t, const int (&es)[4], int n, int k0, int k1,
                                               dd (&out)[4]) {
  const int lane = threadIdx.x & 31;
  dd acc[4] = {};
  const uint16_t* x = p.x + (size_t)t * p.d;
  for (int i8 = k0 / 8 + lane; i8 < k1 / 8; i8 += 32) {
    const uint4 xv = __ldg(reinterpret_cast<const uint4*>(x) + i8);
    const uint32_t xw[4] = {xv.x, xv.y, xv.z, xv.w};
#pragma unroll
    for (int c = 0; c < 4; ++c) {
      if (c >= n) continue;
      const float* w = p.w_router + (size_t)es[c] * p.d;
      const float4 w0 = __ldg(reinterpret_cast<const float4*>(w) + 2 * i8);
      const float4 w1 = __ldg(reinterpret_cast<const float4*>(w) + 2 * i8 + 1);
      const float wv[8] = {w0.x, w0.y, w0.z, w0.w, w1.x, w1.y, w1.z, w1.w};
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        dd_mac(acc[c], __uint_as_float(xw[j] << 16), wv[2 * j]);
        dd_mac(acc[c], __uint_as_float(xw[j] & 0xFFFF0000u), wv[2 * j + 1]);
      }
    }
  }
#pragma unroll
  for (int c = 0; c < 4; ++c) {
    for (int o = 16; o; o >>= 1) acc[c] = dd_add(acc[c], dd_shfl_xor(acc[c], o));
    out[c].hi = __shfl_sync(0xffffffffu, acc[c].hi, 0);
    out[c].lo = __shfl_sync(0xffffffffu, acc[c].lo, 0);
  }
}

// One block per token. (1) fp32 logits (range sums in order, then the bias)
// and their bounds; (2) warp 0: the k-th largest lower bound and the list of
// candidates in index order; (3) every warp: double-float partial logits of the
// candidates over its quarter of d; (4) warp 0: the quarters added in order,
// the bias, k rounds of a warp arg-max over the candidates (value first, then
// the lower expert index), the softmax of the k. The exported logits (hi + lo)
// are the double-float values for the candidates and the fp32 values (lo = 0)
// for the rest.
__global__ void __launch_bounds__(kTopkThreads) topk_kernel(FwdParams p) {
  pdl_enter();
  __shared__ float lf[kTopkMaxE], lb[kTopkMaxE], ub[kTopkMaxE];
  __shared__ short cl[kTopkMaxE];
  __shared__ dd part[kTopkThreads / 32][kTopkMaxE];
  __shared__ int s_nc;
  const int t = blockIdx.x, tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int E = p.E, k = p.k;
  const float up = 1.f + (float)(p.d / 8 + 16) * 0x1p-22f;
  float xs2 = 0.f;
  for (int z = 0; z < p.rsplit; ++z) xs2 += p.xsq[(size_t)z * p.lstride / E + t];
  const float xb = router_gamma(p.d) * 1.01f * (sqrtf(xs2 * up) * up);
  for (int e = tid; e < E; e += kTopkThreads) {
    float l = p.logit_hi[(size_t)t * E + e], ws2 = p.wsq[e];
    for (int z = 1; z < p.rsplit; ++z) {
      l += p.logit_hi[(size_t)z * p.lstride + (size_t)t * E + e];
      ws2 += p.wsq[z * E + e];
    }
    if (p.bias) l += p.bias[e];
    const float beta = fmaf(xb, sqrtf(ws2 * up) * up, 0x1p-22f * fabsf(l)) + 0x1p-126f;
    lf[e] = l;
    lb[e] = l - beta;
    ub[e] = l + beta;
  }
  __syncthreads();
  if (warp == 0) {
    // the k-th largest lower bound (ties: lower index first, for a fixed choice)
    // k rounds over keys of the lower bounds (taken ones retired), each lane's
    // best by selects and the warp's by redux.sync: no divergent branch
    uint32_t taken = 0;
    float kth = -INFINITY;
    const int ni = (E + 31) / 32;
    for (int j = 0; j < k; ++j) {
      unsigned bh = 0, bl = 0;
      int bi = 0x7fffffff;
      for (int i = 0; i < ni; ++i) {
        const int e = 32 * i + lane;
        const unsigned key = (e < E && !((taken >> i) & 1u)) ? fkey(lb[e]) : 0u;
        lane_best_dd(key, 0u, e, bh, bl, bi);
      }
      unsigned mh, ml;
      const int mi = warp_best_dd(bh, bl, bi, mh, ml);
      taken |= ((mi & 31) == lane) ? 1u << (mi >> 5) : 0u;
      kth = unkey(mh);
    }
    int nc = 0;
    for (int i = 0; 32 * i < E; ++i) {
      const int e = 32 * i + lane;
      const bool c = e < E && ub[e] >= kth;
      const unsigned cm = __ballot_sync(0xffffffffu, c);
      if (c) cl[nc + __popc(cm & ((1u << lane) - 1u))] = (short)e;
      nc += __popc(cm);
    }
    if (lane == 0) s_nc = nc;
  }
  __syncthreads();
  const int nc = s_nc;
  {
    // quarter `warp` of d, in whole groups of 8
    const int g8 = p.d / 8, k0 = 8 * (g8 * warp / 4), k1 = 8 * (g8 * (warp + 1) / 4);
    for (int g0 = 0; g0 < nc; g0 += 4) {
      const int n = min(4, nc - g0);
      int es[4];
#pragma unroll
      for (int c = 0; c < 4; ++c) es[c] = c < n ? cl[g0 + c] : 0;
      dd v[4];
      warp_logits_dd(p, t, es, n, k0, k1, v);
      if (lane == 0)
#pragma unroll
        for (int c = 0; c < 4; ++c)
          if (c < n) part[warp][g0 + c] = v[c];
    }
  }
  __syncthreads();
  // the exported logits of the non-candidates: fp32, lo = 0 (candidates below)
  for (int e = tid; e < E; e += kTopkThreads) {
    p.logit_hi[(size_t)t * E + e] = lf[e];
    p.logit_lo[(size_t)t * E + e] = 0.f;
  }
  __syncthreads();
  if (warp != 0) return;
  // candidates c = lane + 32 i: the quarters in order, then the bias
  unsigned kh[kTopkMaxE / 32], kl[kTopkMaxE / 32];  // absent and taken candidates: (0, 0)
  int vid[kTopkMaxE / 32];
#pragma unroll
  for (int i = 0; i < kTopkMaxE / 32; ++i) {
    const int c = lane + 32 * i;
    kh[i] = kl[i] = 0u;
    vid[i] = 0x7fffffff;
    if (c < nc) {
      dd v = part[0][c];
      for (int w = 1; w < kTopkThreads / 32; ++w) v = dd_add(v, part[w][c]);
      const int e = cl[c];
      if (p.bias) v = dd_add(v, dd{p.bias[e], 0.f});
      kh[i] = fkey(v.hi);
      kl[i] = fkey(v.lo);
      vid[i] = e;
      p.logit_hi[(size_t)t * E + e] = v.hi;
      p.logit_lo[(size_t)t * E + e] = v.lo;
    }
  }
  float sel_h = 0.f, sel_l = 0.f;
  int sel_id = 0;
  for (int j = 0; j < k; ++j) {
    unsigned bh = 0, bl = 0;
    int bi = 0x7fffffff;
#pragma unroll
    for (int i = 0; i < kTopkMaxE / 32; ++i) lane_best_dd(kh[i], kl[i], vid[i], bh, bl, bi);
    unsigned mh, ml;
    const int mi = warp_best_dd(bh, bl, bi, mh, ml);
#pragma unroll
    for (int i = 0; i < kTopkMaxE / 32; ++i) {  // expert ids are distinct: one candidate retires
      const bool won = vid[i] == mi;
      kh[i] = won ? 0u : kh[i];
      kl[i] = won ? 0u : kl[i];
      vid[i] = won ? 0x7fffffff : vid[i];
    }
    sel_id = lane == j ? mi : sel_id;
    sel_h = lane == j ? unkey(mh) : sel_h;
    sel_l = lane == j ? unkey(ml) : sel_l;
  }
  const float top_h = __shfl_sync(0xffffffffu, sel_h, 0), top_l = __shfl_sync(0xffffffffu, sel_l, 0);
  float ex = 0.f;
  if (lane < k) ex = expf((sel_h - top_h) + (sel_l - top_l));
  float sum = ex;
  for (int o = 16; o; o >>= 1) sum += __shfl_xor_sync(0xffffffffu, sum, o);
  if (lane < k) {
    p.ids[(size_t)t * k + lane] = sel_id;
    p.gates[(size_t)t * k + lane] = ex / sum;
  }
}

// ---------------------------------------------------------------- router for few tokens
//
// For T <= kRouteDDMaxT the two-pass router above runs on too few blocks to
// use the GPU (its tiles are 32 tokens x 32 experts), and its candidate pass
// is serial per token. Here every logit is a double-float sum (TwoProduct via
// FMA + TwoSum, as in the single-kernel decode path), spread over E x
// ceil(T / kRdTok) blocks: block (e, token group) has 8 warps, warp w sums the
// elements of its eighth of d for up to 8 tokens (lanes stride over groups of
// 8 elements), then a fixed warp tree per token and the 8 warps in order,
// then the bias. The top k are then taken by the bucketing kernel.
constexpr int kRdTok = 8, kRdThreads = 256;

__global__ void __launch_bounds__(kRdThreads) router_dd_kernel(FwdParams p) {
  pdl_enter();
  if ((int)blockIdx.x == p.E) {  // the extra block column: the f16 x of the register-decode GEMMs
    for (int t = blockIdx.y * kRdTok; t < min(p.T, (int)(blockIdx.y + 1) * kRdTok); ++t) {
      prep_x_token(p, t);
      __syncthreads();  // prep_x_token's shared maxima are reused by the next token
    }
    return;
  }
  __shared__ dd part[kRdThreads / 32][kRdTok];
  const int e = blockIdx.x, t0 = blockIdx.y * kRdTok;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int nt = min(kRdTok, p.T - t0);
  const int g8 = p.d / 8, gb = g8 * warp / 8, ge = g8 * (warp + 1) / 8;
  const float4* w4 = reinterpret_cast<const float4*>(p.w_router + (size_t)e * p.d);
  const uint4* x4 = reinterpret_cast<const uint4*>(p.x + (size_t)t0 * p.d);
  dd acc[kRdTok];
#pragma unroll
  for (int j = 0; j < kRdTok; ++j) acc[j] = dd{0.f, 0.f};
  for (int i8 = gb + lane; i8 < ge; i8 += 32) {
    const float4 w0 = __ldg(w4 + 2 * i8), w1 = __ldg(w4 + 2 * i8 + 1);
    const float wv[8] = {w0.x, w0.y, w0.z, w0.w, w1.x, w1.y, w1.z, w1.w};
#pragma unroll
    for (int j = 0; j < kRdTok; ++j) {
      if (j >= nt) break;
      const uint4 xv = __ldg(x4 + (size_t)j * g8 + i8);
      const uint32_t xw[4] = {xv.x, xv.y, xv.z, xv.w};
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        dd_mac(acc[j], __uint_as_float(xw[q] << 16), wv[2 * q]);
        dd_mac(acc[j], __uint_as_float(xw[q] & 0xFFFF0000u), wv[2 * q + 1]);
      }
    }
  }
#pragma unroll
  for (int j = 0; j < kRdTok; ++j) {
    if (j >= nt) break;
    dd v = acc[j];
    for (int o = 16; o; o >>= 1) v = dd_add(v, dd_shfl_xor(v, o));
    if (lane == 0) part[warp][j] = v;
  }
  __syncthreads();
  if (threadIdx.x < nt) {
    const int j = threadIdx.x;
    dd v = part[0][j];
    for (int w = 1; w < kRdThreads / 32; ++w) v = dd_add(v, part[w][j]);
    if (p.bias) v = dd_add(v, dd{p.bias[e], 0.f});
    p.logit_hi[(size_t)(t0 + j) * p.E + e] = v.hi;
    p.logit_lo[(size_t)(t0 + j) * p.E + e] = v.lo;
  }
}

// Top k of token t by one warp from its double-float logits (normalised
// pairs): k rounds of a warp arg-max by (hi, lo, lower index), then the
// softmax of the k selected. NPL = experts per lane.
template <int NPL>
__device__ void topk_warp_dd(const FwdParams& p, int t) {
  const int lane = threadIdx.x & 31, E = p.E, k = p.k;
  unsigned kh[NPL], kl[NPL];  // absent and taken candidates: (0, 0)
#pragma unroll
  for (int i = 0; i < NPL; ++i) {
    const int e = lane + 32 * i;
    kh[i] = e < E ? fkey(p.logit_hi[(size_t)t * E + e]) : 0u;
    kl[i] = e < E ? fkey(p.logit_lo[(size_t)t * E + e]) : 0u;
  }
  float sel_h = 0.f, sel_l = 0.f;
  int sel_id = 0;
  for (int j = 0; j < k; ++j) {
    unsigned bh = 0, bl = 0;
    int bi = 0x7fffffff;
#pragma unroll
    for (int i = 0; i < NPL; ++i) lane_best_dd(kh[i], kl[i], lane + 32 * i, bh, bl, bi);
    unsigned mh, ml;
    const int mi = warp_best_dd(bh, bl, bi, mh, ml);
#pragma unroll
    for (int i = 0; i < NPL; ++i) {
      const bool won = lane + 32 * i == mi;
      kh[i] = won ? 0u : kh[i];
      kl[i] = won ? 0u : kl[i];
    }
    sel_id = lane == j ? mi : sel_id;
    sel_h = lane == j ? unkey(mh) : sel_h;
    sel_l = lane == j ? unkey(ml) : sel_l;
  }
  const float top_h = __shfl_sync(0xffffffffu, sel_h, 0), top_l = __shfl_sync(0xffffffffu, sel_l, 0);
  float ex = 0.f;
  if (lane < k) ex = expf((sel_h - top_h) + (sel_l - top_l));
  float sum = ex;
  for (int o = 16; o; o >>= 1) sum += __shfl_xor_sync(0xffffffffu, sum, o);
  if (lane < k) {
    p.ids[(size_t)t * k + lane] = sel_id;
    p.gates[(size_t)t * k + lane] = ex / sum;
  }
}

// The top k of one token over E <= 512 experts with the whole block (for
// decode-sized calls, where one warp's k rounds over E / 32 logits per lane are
// a long dependent chain): a radix select of the k-th largest logit hi part in
// four 8-bit passes (block histograms), the experts at or above it gathered
// (at most k plus the ones tied on hi with the k-th), then one warp orders
// those few by (hi, lo, lower index) as topk_warp_dd does and forms the gates
// the same way -- the same ids, order and gate bits. More than 32 tied
// candidates (never with continuous logits) fall back to topk_warp_dd.
// `mem` holds 512 words of shared memory.
__device__ void topk_radix_dd(const FwdParams& p, int* mem) {
  const int E = p.E, k = p.k, tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  int* hist = mem;            // [256]
  int* ctl = mem + 256;       // [0] prefix, [1] rank left, [2] candidates
  int* cand = mem + 264;      // [32] candidate experts
  const unsigned key = tid < E ? fkey(p.logit_hi[tid]) : 0u;
  if (tid == 0) {
    ctl[0] = 0;
    ctl[1] = k;
    ctl[2] = 0;
  }
  unsigned prefix = 0u, mask = 0u;
  for (int shift = 24; shift >= 0; shift -= 8) {
    for (int i = tid; i < 256; i += blockDim.x) hist[i] = 0;
    __syncthreads();
    {  // one shared atomic per (warp, bin): most keys share their leading digits
      const bool in = tid < E && (key & mask) == prefix;
      const unsigned act = __ballot_sync(0xffffffffu, in);
      if (in) {
        const unsigned bin = (key >> shift) & 255u;
        const unsigned same = __match_any_sync(act, bin);
        if ((same & ((1u << lane) - 1u)) == 0) atomicAdd(&hist[bin], __popc(same));
      }
    }
    __syncthreads();
    if (warp == 0) {  // the digit of the rank-left-th largest among the keys that match so far
      const int left = ctl[1];
      int c[8], tot = 0;  // lane holds bins 255 - 8 lane - j, from the top
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        c[j] = hist[255 - 8 * lane - j];
        tot += c[j];
      }
      int incl = tot;  // bins above and at this lane's block, counted from the top
      for (int o = 1; o < 32; o <<= 1) {
        const int u = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += u;
      }
      const int above = incl - tot;
      if (above < left && incl >= left) {  // exactly one lane holds the digit
        int run = above;
        for (int j = 0; j < 8; ++j) {
          if (run + c[j] >= left) {
            ctl[0] = (int)((unsigned)ctl[0] | ((unsigned)(255 - 8 * lane - j) << shift));
            ctl[1] = left - run;
            break;
          }
          run += c[j];
        }
      }
    }
    __syncthreads();
    prefix = (unsigned)ctl[0];
    mask |= 255u << shift;
  }
  // the k-th largest hi key is `prefix`: gather every expert at or above it
  {
    const bool in = tid < E && key >= prefix;
    const unsigned act = __ballot_sync(0xffffffffu, in);
    int base = 0;
    if (lane == 0 && act) base = atomicAdd(&ctl[2], __popc(act));
    base = __shfl_sync(0xffffffffu, base, 0);
    const int pos = base + __popc(act & ((1u << lane) - 1u));
    if (in && pos < 32) cand[pos] = tid;
  }
  __syncthreads();
  const int nc = ctl[2];
  if (nc > 32) {  // pathological ties on the hi parts
    if (warp == 0) {
      if (E <= 256) topk_warp_dd<8>(p, 0);
      else topk_warp_dd<16>(p, 0);
    }
    return;
  }
  if (warp != 0) return;
  const int e = lane < nc ? cand[lane] : 0x7fffffff;
  unsigned ckh = lane < nc ? fkey(p.logit_hi[e]) : 0u, ckl = lane < nc ? fkey(p.logit_lo[e]) : 0u;
  int cid = e;
  float sel_h = 0.f, sel_l = 0.f;
  int sel_id = 0;
  for (int j = 0; j < k; ++j) {  // k rounds over one candidate per lane, as topk_warp_dd
    unsigned mh, ml;
    const int mi = warp_best_dd(ckh, ckl, cid, mh, ml);
    const bool won = cid == mi;
    ckh = won ? 0u : ckh;
    ckl = won ? 0u : ckl;
    cid = won ? 0x7fffffff : cid;
    sel_id = lane == j ? mi : sel_id;
    sel_h = lane == j ? unkey(mh) : sel_h;
    sel_l = lane == j ? unkey(ml) : sel_l;
  }
  const float top_h = __shfl_sync(0xffffffffu, sel_h, 0), top_l = __shfl_sync(0xffffffffu, sel_l, 0);
  float ex = 0.f;
  if (lane < k) ex = expf((sel_h - top_h) + (sel_l - top_l));
  float sum = ex;
  for (int o = 16; o; o >>= 1) sum += __shfl_xor_sync(0xffffffffu, sum, o);
  if (lane < k) {
    p.ids[lane] = sel_id;
    p.gates[lane] = ex / sum;
  }
}

// K ranges of the router's fp32 pass: enough blocks for about two per SM.
// Ranges of d for the fp32 pass: about four blocks per SM (measured on the
// 1,024-token layer: 256 blocks -> 512 blocks, 516 -> 506 us per layer; more
// ranges change no rounding count of the certified bound), at most `cap` and
// one per 128-element chunk.
__host__ inline int router_splits(int T, int E, int d, int cap) {
  const int tiles = ((T + kRfTok - 1) / kRfTok) * ((E + kRfExp - 1) / kRfExp);
  const int nch = (d + kRfK - 1) / kRfK;
  int s = (608 + tiles - 1) / tiles;
  s = s < 1 ? 1 : s > cap ? cap : s;
  return s < nch ? s : nch;
}

// ---------------------------------------------------------------- bucketing and work list

constexpr int kBucketThreads = 1024;
constexpr int kBucketChunks = 32;  // warps that count and place the pairs, each over a contiguous chunk
constexpr int kBucketSmem = kBucketChunks * 512 * 4;  // per (chunk, expert) counts, dynamic shared memory

// Exclusive prefix sum over the block (every thread gives v; threads past the
// data give 0); returns the prefix and, in *total, the block's sum.
__device__ __forceinline__ int block_exclusive_scan(int v, int* wsum, int* total) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  int incl = v;
  for (int o = 1; o < 32; o <<= 1) {
    const int u = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += u;
  }
  if (lane == 31) wsum[warp] = incl;
  __syncthreads();
  if (warp == 0) {
    int w = lane < kBucketThreads / 32 ? wsum[lane] : 0;
    for (int o = 1; o < 32; o <<= 1) {
      const int u = __shfl_up_sync(0xffffffffu, w, o);
      if (lane >= o) w += u;
    }
    wsum[lane] = w;  // inclusive over warps
  }
  __syncthreads();
  const int before = warp > 0 ? wsum[warp - 1] : 0;
  *total = wsum[kBucketThreads / 32 - 1];
  __syncthreads();  // wsum is reused by the next scan
  return before + incl - v;
}

// Counting sort of the P = T*k pairs by expert: chunk warps count their
// contiguous range of pairs per expert, a prefix over chunks and one over
// experts give every (chunk, expert) its first position, and the chunk warps
// place their pairs in pair order (ranks within a bucket follow the pair
// index). Then one work-list slot per expert that received pairs (expert
// order) and the shared expert last, from prefix sums of the per-slot unit
// counts.
__global__ void __launch_bounds__(kBucketThreads) bucket_kernel(FwdParams p) {
  pdl_enter();
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, tid = threadIdx.x;
  const int E = p.E, T = p.T, P = p.P;
  extern __shared__ int wc_mem[];
  int (*wc)[512] = reinterpret_cast<int (*)[512]>(wc_mem);  // per (chunk, expert): count, then first position
  __shared__ int wsum[32];
  if (T == 1 && E > 128) {  // one token over many experts: the whole block selects
    topk_radix_dd(p, wc_mem);
    __syncthreads();  // this block's ids writes are visible to the whole block (and wc_mem is free again)
  } else if (T <= kRouteDDMaxT) {  // few tokens: the top k from router_dd_kernel's logits, one warp per token
    if (warp < T) {
      if (E <= 128) topk_warp_dd<4>(p, warp);
      else if (E <= 256) topk_warp_dd<8>(p, warp);
      else topk_warp_dd<16>(p, warp);
    }
    __syncthreads();  // this block's ids writes are visible to the whole block
  }
  // chunk warps: up to kBucketChunks, about 32 pairs each at least (few pairs, few chunks)
  const int nch = max(1, min(kBucketChunks, (P + 31) / 32));
  const int chunk = (P + nch - 1) / nch;
  for (int i = tid; i < nch * E; i += kBucketThreads) wc[i / E][i % E] = 0;
  __syncthreads();
  if (warp < nch) {
    const int q1 = min(P, (warp + 1) * chunk);
    for (int base = warp * chunk; base < q1; base += 32) {
      const int q = base + lane;
      const int e = q < q1 ? p.ids[q] : -1 - lane;
      const unsigned same = __match_any_sync(0xffffffffu, e);
      if (q < q1 && (same & ((1u << lane) - 1u)) == 0) wc[warp][e] += __popc(same);
      __syncwarp();
    }
  }
  __syncthreads();
  int cnt = 0;
  if (tid < E)
    for (int w = 0; w < nch; ++w) {
      const int c = wc[w][tid];
      wc[w][tid] = cnt;
      cnt += c;
    }
  int tot;
  const int off = block_exclusive_scan(tid < E ? cnt : 0, wsum, &tot);
  if (tid < E) {
    p.counts[tid] = cnt;
    p.offsets[tid] = off;
    for (int w = 0; w < nch; ++w) wc[w][tid] += off;
  }
  if (tid == 0) p.offsets[E] = tot;
  __syncthreads();
  if (warp < nch) {
    const int q1 = min(P, (warp + 1) * chunk);
    for (int base = warp * chunk; base < q1; base += 32) {
      const int q = base + lane;
      const bool valid = q < q1;
      const int e = valid ? p.ids[q] : -1 - lane;
      const unsigned same = __match_any_sync(0xffffffffu, e);
      const int rank = __popc(same & ((1u << lane) - 1u));
      const int first = valid ? wc[warp][e] : 0;
      __syncwarp();
      if (valid && rank == 0) wc[warp][e] = first + __popc(same);
      __syncwarp();
      if (valid) {
        const int pos = first + rank;
        p.perm[pos] = q;
        p.inv[q] = pos;
      }
    }
  }
  // work list
  const bool nz = tid < E && cnt > 0 && expert_in_shard(tid, p.e_begin, p.e_end);  // this shard's experts
  // register-decode units: kGemmTiles tiles x kGemmRows rows; affine units: 1 pair tile (gate/up) or
  // kAffDnTiles row tiles (down) x kAffRows rows
  const int rows = p.aff_bits ? kAffRows : kGemmRows, gt = p.aff_bits ? 1 : kGemmTiles,
            dt = p.aff_bits ? kAffDnTiles : kGemmTiles;
  const int blocks = (cnt + rows - 1) / rows, tcb = (cnt + kTcGemmRows - 1) / kTcGemmRows;
  const int ugu = !nz ? 0 : p.tc_gateup ? tcb * tc_gu_pairs(p.F) : blocks * ((p.F / 16 + gt - 1) / gt);
  const int udn = !nz ? 0 : p.tc_gateup ? tcb * tc_dn_pairs(p.d) : blocks * ((p.d / 16 + dt - 1) / dt);
  int ns, gu, dn, pn;
  const int slot = block_exclusive_scan(nz ? 1 : 0, wsum, &ns);
  const int gpre = block_exclusive_scan(ugu, wsum, &gu);
  const int dpre = block_exclusive_scan(udn, wsum, &dn);
  const int ppre = block_exclusive_scan(nz ? tcb : 0, wsum, &pn);
  if (nz) {
    p.slot_expert[slot] = tid;
    p.slot_q0[slot] = off;
    p.slot_n[slot] = cnt;
    p.gu_prefix[slot] = gpre;
    p.dn_prefix[slot] = dpre;
    if (p.tc_gateup) p.panel_prefix[slot] = ppre;
  }
  if (tid == 0) {
    if (p.S > 0 && T > 0 && p.e_begin == 0) {
      p.slot_expert[ns] = E;
      p.slot_q0[ns] = P;
      p.slot_n[ns] = T;
      p.gu_prefix[ns] = gu;
      p.dn_prefix[ns] = dn;
      if (p.tc_gateup) p.panel_prefix[ns] = pn;
      pn += (T + kTcGemmRows - 1) / kTcGemmRows;
      const int sb = (T + rows - 1) / rows;
      gu += p.tc_gateup ? (T + kTcGemmRows - 1) / kTcGemmRows * tc_gu_pairs(p.S) : sb * ((p.S / 16 + gt - 1) / gt);
      dn += p.tc_gateup ? (T + kTcGemmRows - 1) / kTcGemmRows * tc_dn_pairs(p.d) : sb * ((p.d / 16 + dt - 1) / dt);
      ++ns;
    }
    p.gu_prefix[ns] = gu;
    p.dn_prefix[ns] = dn;
    if (p.tc_gateup) p.panel_prefix[ns] = pn;
    *p.n_slots = ns;
  }
}

// ---------------------------------------------------------------- combine

// The shared-expert gate of token t, sigmoid(w_sg . x_t), by a whole block of
// 256 threads: a double-float sum in a fixed order (thread-strided, then a warp
// tree, then the warps in order). Every thread gets the value.
__device__ float shared_gate_block(const FwdParams& p, int t) {
  __shared__ dd red[8];
  __shared__ float g;
  dd acc = dd{0.f, 0.f};
  for (int i = threadIdx.x; i < p.d; i += blockDim.x)
    dd_mac(acc, __uint_as_float((uint32_t)p.x[(size_t)t * p.d + i] << 16), p.w_sg[i]);
  for (int o = 16; o; o >>= 1) acc = dd_add(acc, dd_shfl_xor(acc, o));
  if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = acc;
  __syncthreads();
  if (threadIdx.x == 0) {
    dd z = red[0];
    for (int w = 1; w < (int)(blockDim.x >> 5); ++w) z = dd_add(z, red[w]);
    g = 1.f / (1.f + expf(-(z.hi + z.lo)));
  }
  __syncthreads();
  return g;
}

// y_t = sum_j g_j part_j (pair order) + s_t shared_t, one rounding. A block
// takes 1,024 elements of one token's row (4 per thread, 16-byte loads): the
// token's k (gate, row) pairs are read once into shared memory, then every
// thread's k row loads are independent of each other.
constexpr int kCombineVec = 4;
__global__ void __launch_bounds__(256) combine_kernel(FwdParams p) {
  pdl_enter();
  __shared__ float gk[32];
  __shared__ const float* rk[32];
  const int t = blockIdx.y;
  const float sg = (p.S > 0 && p.w_sg) ? shared_gate_block(p, t) : 1.f;
  if (threadIdx.x < p.k) {  // this shard's pairs only (all of them without sharding); others weigh 0
    const int pj = t * p.k + threadIdx.x;
    const bool mine = expert_in_shard(p.ids[pj], p.e_begin, p.e_end);
    gk[threadIdx.x] = mine ? p.gates[pj] : 0.f;
    rk[threadIdx.x] = mine ? p.part + (size_t)p.inv[pj] * p.d : nullptr;
  }
  __syncthreads();
  const int r = (blockIdx.x * blockDim.x + threadIdx.x) * kCombineVec;
  if (r >= p.d) return;
  float acc[kCombineVec] = {0.f, 0.f, 0.f, 0.f};
  for (int j = 0; j < p.k; ++j) {
    if (!rk[j]) continue;
    const float4 v = *reinterpret_cast<const float4*>(rk[j] + r);
    const float g = gk[j];
    acc[0] = fmaf(g, v.x, acc[0]);
    acc[1] = fmaf(g, v.y, acc[1]);
    acc[2] = fmaf(g, v.z, acc[2]);
    acc[3] = fmaf(g, v.w, acc[3]);
  }
  if (p.S > 0 && p.e_begin == 0) {
    const float4 v = *reinterpret_cast<const float4*>(p.part + (size_t)(p.P + t) * p.d + r);
    acc[0] += sg * v.x;
    acc[1] += sg * v.y;
    acc[2] += sg * v.z;
    acc[3] += sg * v.w;
  }
  if (p.out_f32) {
    *reinterpret_cast<float4*>(reinterpret_cast<float*>(p.out) + (size_t)t * p.d + r) =
        make_float4(acc[0], acc[1], acc[2], acc[3]);
  } else {
    __nv_bfloat16* o = reinterpret_cast<__nv_bfloat16*>(p.out) + (size_t)t * p.d + r;
    *reinterpret_cast<__nv_bfloat162*>(o) = __floats2bfloat162_rn(acc[0], acc[1]);
    *reinterpret_cast<__nv_bfloat162*>(o + 2) = __floats2bfloat162_rn(acc[2], acc[3]);
  }
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

void launch_router(FwdParams p, cudaStream_t stream, bool with_prep_x) {
  if (p.T <= kRouteDDMaxT) {  // the top k follow in bucket_kernel; one more block column prepares x if asked
    launch_chained(router_dd_kernel, dim3(p.E + (with_prep_x ? 1 : 0), (p.T + kRdTok - 1) / kRdTok), dim3(kRdThreads),
                   0, stream, p);
    return;
  }
  p.rsplit = router_splits(p.T, p.E, p.d, p.rsplit_max > 0 ? p.rsplit_max : kRouterSplits);
  launch_chained(router_fp32_kernel, dim3((p.T + kRfTok - 1) / kRfTok, (p.E + kRfExp - 1) / kRfExp, p.rsplit),
                 dim3(kRfThreads), 0, stream, p);
  launch_chained(topk_kernel, dim3(p.T), dim3(kTopkThreads), 0, stream, p);
}

cudaError_t configure_kernels() {
  return cudaFuncSetAttribute(bucket_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kBucketSmem);
}

const char* const kForwardPhaseNames = "route,gateup,down,combine";
const char* const kForwardPhaseNamesTc = "route,panels,gateup,down,combine";

cudaError_t launch_forward(const FwdParams& p, cudaStream_t stream, int num_sms, cudaEvent_t const* events) {
  if (p.T == 0) return cudaSuccess;
  int ev = 0;
  auto mark = [&]() {
    if (events) cudaEventRecord(events[ev++], stream);
  };
  mark();
  // f16 x of the register-decode and affine GEMMs: inside the router launch for T <= kRouteDDMaxT
  if (!p.tc_gateup && p.T > kRouteDDMaxT) launch_chained(prep_x_kernel, dim3(p.T), dim3(256), 0, stream, p);
  launch_router(p, stream, !p.tc_gateup);
  launch_chained(bucket_kernel, dim3(1), dim3(kBucketThreads), kBucketSmem, stream, p);
  mark();
  cudaError_t e = cudaSuccess;
  if (p.tc_gateup) {
    if ((e = launch_panels_tc(p, stream)) != cudaSuccess) return e;
    mark();
  }
  e = p.aff_bits    ? launch_affine_gateup(p, stream, num_sms)
      : p.tc_gateup ? launch_gemm_gateup_tc(p, stream, num_sms)
                    : launch_gemm_gateup(p, stream, num_sms);
  if (e != cudaSuccess) return e;
  mark();
  e = p.aff_bits    ? launch_affine_down(p, stream, num_sms)
      : p.tc_gateup ? launch_gemm_down_tc(p, stream, num_sms)
                    : launch_gemm_down(p, stream, num_sms);
  if (e != cudaSuccess) return e;
  mark();
  launch_chained(combine_kernel, dim3((p.d / kCombineVec + 255) / 256, p.T), dim3(256), 0, stream, p);
  mark();
  return cudaGetLastError();
}

cudaError_t launch_route(const FwdParams& p, cudaStream_t stream) {
  if (p.T == 0) return cudaSuccess;
  launch_router(p, stream, false);
  launch_chained(bucket_kernel, dim3(1), dim3(kBucketThreads), kBucketSmem, stream, p);
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
