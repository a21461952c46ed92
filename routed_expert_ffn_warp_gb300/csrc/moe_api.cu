// Host side of the routed-expert FFN library: context, loads, forward, debug
// exports. The C ABI is declared in include/moe.h.
#include <cuda.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <cstdio>
#include <cstring>
#include <string>

#include "../../include/moe.h"
#include "moe_internal.h"

struct moe_ctx {
  moe_config cfg{};
  int device = 0;
  int num_sms = 0;
  bool router_loaded = false;
  bool experts_loaded = false;
  std::string err;
  // weights
  uint8_t* packed = nullptr;
  size_t packed_bytes = 0;
  size_t expert_stride = 0;
  uint8_t* tcw = nullptr;  // gate/up copy for the tcgen05 GEMM (MOE_FLAG_TC_GATEUP)
  size_t tcw_bytes = 0;
  size_t tcw_stride = 0;
  uint8_t* tcwd = nullptr;  // down copy for the tcgen05 GEMM
  size_t tcwd_bytes = 0;
  size_t tcwd_stride = 0;
  CUtensorMap tmap_gu{};  // tensor maps the tcgen05 kernels load tcw / tcwd through (tile pairs)
  CUtensorMap tmap_dn{};
  CUtensorMap tmap_gu3{};  // 3-D maps whose box is a whole tile-pair block (codes + scale bytes)
  CUtensorMap tmap_dn3{};
  float* w_router = nullptr;
  float* bias = nullptr;
  bool has_bias = false;
  float* w_sg = nullptr;  // shared-expert gate row [d] (contexts with a shared expert)
  bool has_sg = false;
  // workspace (one allocation, zeroed at create)
  void* ws = nullptr;
  size_t ws_bytes = 0;
  moe::FwdParams base{};
  void* x_dev = nullptr;    // host-API staging of x
  void* out_dev = nullptr;  // host-API staging of out
  int* load_err = nullptr;  // repack NaN-scale flag
  int last_T = 0;
  cudaEvent_t prof[moe::kForwardPhasesTc + 1] = {};
  int n_prof = 0;
  int max_smem = 0;
  bool decode_ok = false;    // the fused mma.sync kernel serves T <= 16 (contexts with the packed copy)
  bool fused_tc_ok = false;  // the fused tcgen05 kernel serves T <= 16 (contexts with the tcgen05 copies)
  moe::DecParams dec{};
  moe::TcLayerParams tcl{};
};

namespace {

std::string g_create_error;

// Makes ctx's device current for the duration of a call and restores the
// caller's device afterwards.
struct DeviceGuard {
  int prev = -1;
  bool ok = true;
  explicit DeviceGuard(int dev) {
    if (cudaGetDevice(&prev) != cudaSuccess) prev = -1;
    if (prev != dev) ok = cudaSetDevice(dev) == cudaSuccess;
  }
  ~DeviceGuard() {
    int cur = -1;
    if (prev >= 0 && cudaGetDevice(&cur) == cudaSuccess && cur != prev) cudaSetDevice(prev);
  }
};

int fail(moe_ctx* ctx, int code, const std::string& msg) {
  if (ctx) ctx->err = msg;
  else g_create_error = msg;
  return code;
}

int cuda_fail(moe_ctx* ctx, cudaError_t e, const char* what) {
  return fail(ctx, MOE_ERR_CUDA, std::string(what) + ": " + cudaGetErrorString(e));
}

size_t align_up(size_t v, size_t a) { return (v + a - 1) / a * a; }

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// Address at which the current device reaches host buffer p, if p is
// page-locked memory mapped into its address space (cudaHostAlloc /
// cudaMallocHost under unified addressing, cudaHostRegister with the mapped
// flag); nullptr for pageable or unmapped memory.
const void* mapped_host_address(const void* p) {
  cudaPointerAttributes a{};
  if (cudaPointerGetAttributes(&a, p) != cudaSuccess) {
    cudaGetLastError();  // the query failed: not an error of this call
    return nullptr;
  }
  return a.type == cudaMemoryTypeHost ? a.devicePointer : nullptr;
}

// A single-launch path serves T <= 16 when its plan fits: the tcgen05 kernel
// for contexts with the tcgen05 weight copies, the mma.sync kernel for those
// with the packed copy (MOE_FLAG_NO_TC).
bool uses_decode(const moe_ctx* ctx, int T) {
  return T > 0 && T <= moe::kDecodeMaxT && (ctx->fused_tc_ok || ctx->decode_ok);
}

}  // namespace

extern "C" {

int moe_create(const moe_config* cfg, int device, moe_ctx** out) {
  if (!out) return fail(nullptr, MOE_ERR_INVALID_ARG, "out is NULL");
  *out = nullptr;
  if (!cfg) return fail(nullptr, MOE_ERR_INVALID_ARG, "cfg is NULL");
  const moe_config& c = *cfg;
  const bool all_experts = c.expert_begin == 0 && c.expert_end == 0;
  if (c.d <= 0 || c.d % 32 || c.ffn <= 0 || c.ffn % 32 || c.shared_ffn < 0 || c.shared_ffn % 32 ||
      (!all_experts && (c.expert_begin < 0 || c.expert_begin >= c.expert_end || c.expert_end > c.n_experts)) ||
      c.n_experts < 1 || c.n_experts > 512 || c.top_k < 1 || c.top_k > c.n_experts || c.top_k > 32 ||
      c.t_max < 0 || c.t_max > 65536 || (c.out_dtype != MOE_OUT_BF16 && c.out_dtype != MOE_OUT_F32) ||
      (c.flags & ~(unsigned)(MOE_FLAG_TEST_FORCE_TIMEOUT | MOE_FLAG_GENERAL_PATH | MOE_FLAG_TC_GATEUP | MOE_FLAG_NO_TC)) ||
      ((c.flags & MOE_FLAG_TC_GATEUP) && (c.flags & MOE_FLAG_NO_TC)) ||
      (c.weight_format != MOE_FORMAT_MXFP4 && c.weight_format != MOE_FORMAT_AFFINE64))
    return fail(nullptr, MOE_ERR_INVALID_ARG,
                "config out of range (d, ffn, shared_ffn multiples of 32; 1 <= E <= 512; 1 <= k <= min(E, 32); "
                "0 <= t_max <= 65536; out_dtype 0/1; known flags, not both TC_GATEUP and NO_TC; "
                "0 <= expert_begin < expert_end <= E or both 0; a known weight_format)");
  const bool affine = c.weight_format == MOE_FORMAT_AFFINE64;
  if (affine && (!moe::affine_bits_supported(c.weight_bits) || c.d % 64 || c.ffn % 64 || c.shared_ffn % 64 ||
                 (c.flags & MOE_FLAG_TC_GATEUP)))
    return fail(nullptr, MOE_ERR_INVALID_ARG,
                "affine experts need weight_bits 2, 3, 4 or 8, d, ffn and shared_ffn multiples of 64, and no "
                "MOE_FLAG_TC_GATEUP");
  moe_ctx* ctx = new (std::nothrow) moe_ctx();
  if (!ctx) return fail(nullptr, MOE_ERR_NOMEM, "host allocation failed");
  ctx->cfg = c;
  ctx->device = device;
  DeviceGuard guard(device);
  if (!guard.ok) {
    delete ctx;
    return fail(nullptr, MOE_ERR_CUDA, "cudaSetDevice failed");
  }
  cudaError_t e = cudaDeviceGetAttribute(&ctx->num_sms, cudaDevAttrMultiProcessorCount, device);
  if (e == cudaSuccess) e = cudaDeviceGetAttribute(&ctx->max_smem, cudaDevAttrMaxSharedMemoryPerBlockOptin, device);
  if (e != cudaSuccess) {
    delete ctx;
    return fail(nullptr, MOE_ERR_CUDA, std::string("cudaDeviceGetAttribute: ") + cudaGetErrorString(e));
  }
  const int d = c.d, F = c.ffn, E = c.n_experts, k = c.top_k, S = c.shared_ffn, Tm = std::max(c.t_max, 1);
  const int eb = all_experts ? 0 : c.expert_begin, ee = all_experts ? E : c.expert_end;
  const int El = ee - eb;                   // routed experts this context holds
  const bool Sl = S > 0 && eb == 0;         // ... and the shared expert
  const int abits = affine ? c.weight_bits : 0;
  ctx->expert_stride = affine ? moe::aff_expert_bytes(d, F, abits) : moe::expert_packed_bytes(d, F);
  const bool tc_fits =
      std::max(moe::tc_gemm_smem_bytes(E, false), moe::tc_gemm_smem_bytes(E, true)) <= (size_t)ctx->max_smem;
  if ((c.flags & MOE_FLAG_TC_GATEUP) && !tc_fits) {
    delete ctx;
    return fail(nullptr, MOE_ERR_INVALID_ARG, "too many experts for the tcgen05 GEMM's shared-memory tables");
  }
  // One weight copy per context. Contexts whose calls can reach more than
  // kFusedMaxPairs (token, expert) pairs keep the tcgen05 block layout (the fused
  // tcgen05 kernel for T <= 16, the tcgen05 GEMMs above); smaller ones -- every
  // call a few tokens, where the fused mma.sync kernel is the faster -- keep the
  // packed tiles. MOE_FLAG_TC_GATEUP / MOE_FLAG_NO_TC force either.
  // Affine contexts keep their own tiles (the packed pointer) and always take the multi-kernel path.
  const bool tc = !affine && ((c.flags & MOE_FLAG_TC_GATEUP) ||
                              (!(c.flags & MOE_FLAG_NO_TC) && tc_fits && (long long)c.t_max * k > moe::kFusedMaxPairs));
  if (!tc)
    ctx->packed_bytes = ctx->expert_stride * (size_t)El +
                        (Sl ? (affine ? moe::aff_expert_bytes(d, S, abits) : moe::expert_packed_bytes(d, S)) : 0);
  if (tc) {
    ctx->tcw_stride = moe::tc_expert_bytes(d, F);
    ctx->tcw_bytes = ctx->tcw_stride * (size_t)El + (Sl ? moe::tc_expert_bytes(d, S) : 0);
    ctx->tcwd_stride = moe::tc_down_bytes(d, F);
    ctx->tcwd_bytes = ctx->tcwd_stride * (size_t)El + (Sl ? moe::tc_down_bytes(d, S) : 0);
  }

  const size_t Pm = (size_t)Tm * k, Qm = Pm + (S > 0 ? (size_t)Tm : 0);
  const int d64 = moe::k64_tiles(d) * 64;
  const int fmax64 = moe::k64_tiles(std::max(F, S)) * 64;
  const int hgroups = fmax64 / 16;
  size_t off = 0;
  auto take = [&](size_t bytes) {
    size_t o = off;
    off = align_up(off + bytes, 256);
    return o;
  };
  const size_t o_x16 = take((size_t)Tm * d64 * 2), o_xinv = take((size_t)Tm * 4);
  const int xq_spitch = (d64 / 32 + 3) / 4 * 4;
  const size_t o_xq = take((size_t)Tm * 2 * d64), o_xqs = take((size_t)Tm * 2 * xq_spitch);
  const size_t o_lh = take((size_t)moe::kRouterSplits * Tm * E * 4);
  const size_t o_xsq = take((size_t)moe::kRouterSplits * Tm * 4), o_wsq = take((size_t)moe::kRouterSplits * E * 4);
  const size_t o_ids = take(Pm * 4), o_gates = take(Pm * 4), o_counts = take((size_t)E * 4),
               o_offsets = take((size_t)(E + 1) * 4), o_perm = take(Pm * 4), o_inv = take(Pm * 4);
  const size_t o_ns = take(4), o_se = take((size_t)(E + 1) * 4), o_sq = take((size_t)(E + 1) * 4),
               o_sn = take((size_t)(E + 1) * 4), o_gp = take((size_t)(E + 2) * 4), o_dp = take((size_t)(E + 2) * 4);
  // activation panels of the tcgen05 GEMM: at most ceil(Q / 48) + slots blocks
  const size_t n_panels = tc ? Qm / moe::kTcGemmRows + (size_t)E + 2 : 0;
  const size_t o_panel = take(n_panels * moe::tc_ksteps(d) * moe::kTcPanelStep), o_pp = take((size_t)(E + 2) * 4);
  const size_t o_hpanel = take(n_panels * moe::tc_ksteps(std::max(F, S)) * moe::kTcPanelStepD);
  const size_t o_h = take(Qm * 2 * fmax64 * 2), o_hs = take(Qm * hgroups * 4), o_part = take(Qm * d * 4);
  const size_t o_xd = take((size_t)Tm * d * 2), o_od = take((size_t)Tm * d * (c.out_dtype == MOE_OUT_F32 ? 4 : 2));
  const size_t o_status = take(4), o_lerr = take(4);
  // affine experts: group sums of x (per 64) and of h (per 16)
  const int xg_pitch = (d / 64 + 3) / 4 * 4;
  const size_t o_xg = take(affine ? (size_t)Tm * xg_pitch * 4 : 0), o_hb = take(affine ? Qm * hgroups * 4 : 0);
  // a row of zeros that absent activation rows of the affine GEMMs read (never written)
  const size_t o_zero = take(affine ? (size_t)4 * std::max(d64, fmax64) : 0);
  // fused mma.sync path: launch-tagged words of h, its scales and the partial down rows
  const size_t Qd = (size_t)std::min(Tm, moe::kDecodeMaxT) * (k + (S > 0 ? 1 : 0));  // pair rows of the fused path
  const size_t o_hw = take(Qd * fmax64 * 8), o_hsw = take(Qd * hgroups * 8), o_pw = take(Qd * d * 8),
               o_bar = take((size_t)std::max(ctx->num_sms, 1) * 4),
               o_lw = take((size_t)moe::kLogitWordCopies * std::min(Tm, moe::kDecodeMaxT) * (E + 1) * 2 * 8);
  // fused tcgen05 path: x planes and h planes per K step with their launch-tagged flags, row-tile counters
  const int tcap = std::min(Tm, moe::kDecodeMaxT), npad = tcap <= 8 ? 8 : (tcap + 7) & ~7;
  const int xp_step = 2 * npad * 128 + 512, hp_step = 4 * npad * 128 + 512, hp_ks = moe::tc_ksteps(std::max(F, S));
  const int max_slots = std::min(E, tcap * k) + (S > 0 ? 1 : 0);
  const size_t o_xpl = take(tc ? (size_t)moe::tc_ksteps(d) * xp_step : 0), o_xfl = take(tc ? (size_t)moe::tc_ksteps(d) * 4 : 0),
               o_hpl = take(tc ? (size_t)max_slots * hp_ks * hp_step : 0), o_hfl = take(tc ? (size_t)max_slots * hp_ks * 4 : 0),
               o_dcnt = take((size_t)2 * moe::tc_dtiles(d) * 4);
  ctx->ws_bytes = off;

  if ((tc && (e = cudaMalloc(&ctx->tcw, ctx->tcw_bytes)) != cudaSuccess) ||
      (tc && (e = cudaMalloc(&ctx->tcwd, ctx->tcwd_bytes)) != cudaSuccess) ||
      (!tc && (e = cudaMalloc(&ctx->packed, ctx->packed_bytes)) != cudaSuccess) ||
      (e = cudaMalloc(&ctx->w_router, (size_t)E * d * 4)) != cudaSuccess ||
      (e = cudaMalloc(&ctx->bias, (size_t)E * 4)) != cudaSuccess ||
      (S > 0 && (e = cudaMalloc(&ctx->w_sg, (size_t)d * 4)) != cudaSuccess) ||
      (e = cudaMalloc(&ctx->ws, ctx->ws_bytes)) != cudaSuccess) {
    moe_destroy(ctx);
    return fail(nullptr, MOE_ERR_NOMEM, std::string("cudaMalloc: ") + cudaGetErrorString(e));
  }
  if (tc && (!moe::encode_tc_weight_map(ctx->tcw, ctx->tcw_bytes, &ctx->tmap_gu, 256) ||
             !moe::encode_tc_weight_map(ctx->tcwd, ctx->tcwd_bytes, &ctx->tmap_dn, 256) ||
             !moe::encode_tc_block_map(ctx->tcw, ctx->tcw_bytes, &ctx->tmap_gu3) ||
             !moe::encode_tc_block_map(ctx->tcwd, ctx->tcwd_bytes, &ctx->tmap_dn3))) {
    moe_destroy(ctx);
    return fail(nullptr, MOE_ERR_CUDA, "cuTensorMapEncodeTiled refused the tcgen05 weight copy");
  }
  if ((e = cudaMemset(ctx->ws, 0, ctx->ws_bytes)) != cudaSuccess ||
      (e = cudaMemset(ctx->bias, 0, (size_t)E * 4)) != cudaSuccess) {
    moe_destroy(ctx);
    return fail(nullptr, MOE_ERR_CUDA, std::string("cudaMemset: ") + cudaGetErrorString(e));
  }
  char* w = static_cast<char*>(ctx->ws);
  moe::FwdParams& p = ctx->base;
  p.d = d;
  p.F = F;
  p.E = E;
  p.e_begin = eb;
  p.e_end = ee;
  p.k = k;
  p.S = S;
  p.d64 = d64;
  p.fmax64 = fmax64;
  p.hgroups = hgroups;
  p.out_f32 = c.out_dtype == MOE_OUT_F32;
  p.tc_gateup = tc ? 1 : 0;
  p.w_router = ctx->w_router;
  p.bias = nullptr;
  p.packed = ctx->packed;
  p.expert_stride = ctx->expert_stride;
  p.aff_bits = abits;
  p.xgsum = affine ? reinterpret_cast<float*>(w + o_xg) : nullptr;
  p.xg_pitch = xg_pitch;
  p.hbsum = affine ? reinterpret_cast<float*>(w + o_hb) : nullptr;
  p.zeros = affine ? w + o_zero : nullptr;
  p.x16 = reinterpret_cast<uint16_t*>(w + o_x16);
  p.xinv = reinterpret_cast<float*>(w + o_xinv);
  p.tcw = ctx->tcw;
  p.tcw_stride = ctx->tcw_stride;
  p.xpanel = reinterpret_cast<uint8_t*>(w + o_panel);
  p.tcwd = ctx->tcwd;
  p.tcwd_stride = ctx->tcwd_stride;
  p.hpanel = reinterpret_cast<uint8_t*>(w + o_hpanel);
  p.tmap_gu = &ctx->tmap_gu;
  p.tmap_dn = &ctx->tmap_dn;
  p.tmap_gu3 = &ctx->tmap_gu3;
  p.tmap_dn3 = &ctx->tmap_dn3;
  p.panel_prefix = reinterpret_cast<int32_t*>(w + o_pp);
  p.xq = reinterpret_cast<uint8_t*>(w + o_xq);
  p.xqs = reinterpret_cast<uint8_t*>(w + o_xqs);
  p.xq_spitch = xq_spitch;
  p.logit_hi = reinterpret_cast<float*>(w + o_lh);
  p.lstride = (size_t)Tm * E;
  p.logit_lo = p.logit_hi + p.lstride;
  p.xsq = reinterpret_cast<float*>(w + o_xsq);
  p.wsq = reinterpret_cast<float*>(w + o_wsq);
  p.ids = reinterpret_cast<int32_t*>(w + o_ids);
  p.gates = reinterpret_cast<float*>(w + o_gates);
  p.counts = reinterpret_cast<int32_t*>(w + o_counts);
  p.offsets = reinterpret_cast<int32_t*>(w + o_offsets);
  p.perm = reinterpret_cast<int32_t*>(w + o_perm);
  p.inv = reinterpret_cast<int32_t*>(w + o_inv);
  p.n_slots = reinterpret_cast<int32_t*>(w + o_ns);
  p.slot_expert = reinterpret_cast<int32_t*>(w + o_se);
  p.slot_q0 = reinterpret_cast<int32_t*>(w + o_sq);
  p.slot_n = reinterpret_cast<int32_t*>(w + o_sn);
  p.gu_prefix = reinterpret_cast<int32_t*>(w + o_gp);
  p.dn_prefix = reinterpret_cast<int32_t*>(w + o_dp);
  p.hbuf = reinterpret_cast<uint16_t*>(w + o_h);
  p.hscale = reinterpret_cast<float*>(w + o_hs);
  p.part = reinterpret_cast<float*>(w + o_part);
  p.status = reinterpret_cast<int*>(w + o_status);
  ctx->x_dev = w + o_xd;
  ctx->out_dev = w + o_od;
  ctx->load_err = reinterpret_cast<int*>(w + o_lerr);
  moe::DecParams& dp = ctx->dec;
  dp.f = p;
  dp.hwords = reinterpret_cast<unsigned long long*>(w + o_hw);
  dp.hswords = reinterpret_cast<unsigned long long*>(w + o_hsw);
  dp.pwords = reinterpret_cast<unsigned long long*>(w + o_pw);
  dp.bar_flags = reinterpret_cast<unsigned*>(w + o_bar);
  dp.lwords = reinterpret_cast<unsigned long long*>(w + o_lw);
  dp.tcap = std::min(Tm, moe::kDecodeMaxT);
  dp.wait_ns = 50000000LL;  // 50 ms: orders of magnitude above a layer's runtime
  dp.test_extra = (c.flags & MOE_FLAG_TEST_FORCE_TIMEOUT) ? 1 : 0;
  dp.test_wait_ns = 2000000LL;  // 2 ms
  // kernel attributes are per device: set them with this context's device current
  if ((e = moe::configure_decode(ctx->max_smem)) != cudaSuccess || (e = moe::configure_tcgemm(ctx->max_smem)) != cudaSuccess ||
      (e = moe::configure_gemm()) != cudaSuccess || (e = moe::configure_affine()) != cudaSuccess ||
      (e = moe::configure_kernels()) != cudaSuccess) {
    moe_destroy(ctx);
    return fail(nullptr, MOE_ERR_CUDA, std::string("cudaFuncSetAttribute: ") + cudaGetErrorString(e));
  }
  // The fused kernel's CTAs wait on each other (bounded): it is used only when
  // one CTA per SM fits, so that a grid of one CTA per SM can be resident at once.
  if (tc && (e = moe::configure_tc_layer(ctx->max_smem)) != cudaSuccess) {
    moe_destroy(ctx);
    return fail(nullptr, MOE_ERR_CUDA, std::string("cudaFuncSetAttribute: ") + cudaGetErrorString(e));
  }
  const bool single = !(c.flags & MOE_FLAG_GENERAL_PATH);
  if (tc) {
    moe::TcLayerParams& tp = ctx->tcl;
    tp.d = dp;
    tp.xplane = reinterpret_cast<uint8_t*>(w + o_xpl);
    tp.xflag = reinterpret_cast<unsigned*>(w + o_xfl);
    tp.hpanel = reinterpret_cast<uint8_t*>(w + o_hpl);
    tp.hflag = reinterpret_cast<unsigned*>(w + o_hfl);
    tp.dcnt = reinterpret_cast<int*>(w + o_dcnt);
    tp.hp_ksteps = hp_ks;
    tp.max_slots = max_slots;
    ctx->fused_tc_ok = single && moe::tc_layer_plan(tp, ctx->max_smem, ctx->num_sms) && tp.xp_step == xp_step &&
                       tp.hp_step == hp_step && moe::tc_layer_blocks_per_sm(tp) >= 1;
  } else if (!affine) {
    ctx->decode_ok = single && moe::decode_plan(dp, ctx->max_smem, ctx->num_sms) && moe::decode_blocks_per_sm(dp) >= 1;
  }
  *out = ctx;
  return MOE_OK;
}

int moe_load_router(moe_ctx* ctx, const float* wr, const float* bias) {
  if (!ctx) return MOE_ERR_INVALID_ARG;
  if (!wr) return fail(ctx, MOE_ERR_INVALID_ARG, "router weights are NULL");
  DeviceGuard guard(ctx->device);
  const size_t n = (size_t)ctx->cfg.n_experts * ctx->cfg.d;
  cudaError_t e = cudaMemcpy(ctx->w_router, wr, n * 4, cudaMemcpyDefault);
  if (e != cudaSuccess) return cuda_fail(ctx, e, "router copy");
  if (bias) {
    e = cudaMemcpy(ctx->bias, bias, (size_t)ctx->cfg.n_experts * 4, cudaMemcpyDefault);
    if (e != cudaSuccess) return cuda_fail(ctx, e, "bias copy");
  }
  ctx->has_bias = bias != nullptr;
  ctx->base.bias = ctx->has_bias ? ctx->bias : nullptr;
  ctx->router_loaded = true;
  return MOE_OK;
}

int moe_load_shared_gate(moe_ctx* ctx, const float* w) {
  if (!ctx) return MOE_ERR_INVALID_ARG;
  if (ctx->cfg.shared_ffn <= 0) return fail(ctx, MOE_ERR_INVALID_ARG, "the context has no shared expert to gate");
  if (!w) {
    ctx->has_sg = false;
    return MOE_OK;
  }
  DeviceGuard guard(ctx->device);
  const cudaError_t e = cudaMemcpy(ctx->w_sg, w, (size_t)ctx->cfg.d * 4, cudaMemcpyDefault);
  if (e != cudaSuccess) return cuda_fail(ctx, e, "shared gate copy");
  ctx->has_sg = true;
  return MOE_OK;
}

int moe_load_experts(moe_ctx* ctx, const uint8_t* codes, const uint8_t* scales) {
  if (!ctx) return MOE_ERR_INVALID_ARG;
  if (!codes || !scales) return fail(ctx, MOE_ERR_INVALID_ARG, "codes or scales are NULL");
  if (ctx->base.aff_bits)
    return fail(ctx, MOE_ERR_INVALID_ARG, "the context holds affine experts: load them with moe_load_experts_affine");
  DeviceGuard guard(ctx->device);
  const int d = ctx->cfg.d, F = ctx->cfg.ffn;
  const int E = ctx->base.e_end - ctx->base.e_begin;                 // routed experts the context holds
  const int S = ctx->base.e_begin == 0 ? ctx->cfg.shared_ffn : 0;  // its shared expert, if any
  const size_t ccs = (size_t)3 * F * d / 2, css = (size_t)3 * F * d / 32;  // canonical strides
  const size_t chunk_bytes = (size_t)256 << 20;
  const int per_chunk = (int)std::max<size_t>(1, chunk_bytes / ccs);
  const size_t stage_c = std::max(ccs * (size_t)std::min(per_chunk, E), S > 0 ? (size_t)3 * S * d / 2 : 0);
  const size_t stage_s = std::max(css * (size_t)std::min(per_chunk, E), S > 0 ? (size_t)3 * S * d / 32 : 0);
  uint8_t* sc = nullptr;
  uint8_t* ss = nullptr;
  cudaError_t e = cudaMalloc(&sc, stage_c);
  if (e == cudaSuccess) e = cudaMalloc(&ss, stage_s);
  if (e != cudaSuccess) {
    cudaFree(sc);
    return fail(ctx, MOE_ERR_NOMEM, std::string("staging cudaMalloc: ") + cudaGetErrorString(e));
  }
  int rc = MOE_OK;
  e = cudaMemset(ctx->load_err, 0, 4);
  for (int x0 = 0; x0 < E && e == cudaSuccess; x0 += per_chunk) {
    const int n = std::min(per_chunk, E - x0);
    if ((e = cudaMemcpy(sc, codes + (size_t)x0 * ccs, ccs * n, cudaMemcpyDefault)) != cudaSuccess) break;
    if ((e = cudaMemcpy(ss, scales + (size_t)x0 * css, css * n, cudaMemcpyDefault)) != cudaSuccess) break;
    if (ctx->packed && (e = moe::launch_repack(sc, ss, n, d, F, ccs, css, ctx->packed + (size_t)x0 * ctx->expert_stride,
                                               ctx->expert_stride, ctx->load_err, 0)) != cudaSuccess)
      break;
    if (ctx->tcw && (e = moe::launch_repack_tc(sc, ss, n, d, F, ccs, css, ctx->tcw + (size_t)x0 * ctx->tcw_stride,
                                               ctx->tcw_stride, false, ctx->load_err, 0)) != cudaSuccess)
      break;
    if (ctx->tcwd && (e = moe::launch_repack_tc(sc, ss, n, d, F, ccs, css, ctx->tcwd + (size_t)x0 * ctx->tcwd_stride,
                                                ctx->tcwd_stride, true, ctx->load_err, 0)) != cudaSuccess)
      break;
    e = cudaDeviceSynchronize();
  }
  if (e == cudaSuccess && S > 0) {
    const size_t sc_b = (size_t)3 * S * d / 2, ss_b = (size_t)3 * S * d / 32;
    if ((e = cudaMemcpy(sc, codes + (size_t)E * ccs, sc_b, cudaMemcpyDefault)) == cudaSuccess &&
        (e = cudaMemcpy(ss, scales + (size_t)E * css, ss_b, cudaMemcpyDefault)) == cudaSuccess &&
        (!ctx->packed || (e = moe::launch_repack(sc, ss, 1, d, S, sc_b, ss_b, ctx->packed + (size_t)E * ctx->expert_stride,
                                                 moe::expert_packed_bytes(d, S), ctx->load_err, 0)) == cudaSuccess) &&
        (!ctx->tcw || (e = moe::launch_repack_tc(sc, ss, 1, d, S, sc_b, ss_b, ctx->tcw + (size_t)E * ctx->tcw_stride,
                                                 moe::tc_expert_bytes(d, S), false, ctx->load_err, 0)) == cudaSuccess) &&
        (!ctx->tcwd || (e = moe::launch_repack_tc(sc, ss, 1, d, S, sc_b, ss_b, ctx->tcwd + (size_t)E * ctx->tcwd_stride,
                                                  moe::tc_down_bytes(d, S), true, ctx->load_err, 0)) == cudaSuccess))
      e = cudaDeviceSynchronize();
  }
  int nan_flag = 0;
  if (e == cudaSuccess) e = cudaMemcpy(&nan_flag, ctx->load_err, 4, cudaMemcpyDeviceToHost);
  cudaFree(sc);
  cudaFree(ss);
  if (e != cudaSuccess) return cuda_fail(ctx, e, "expert load");
  if (nan_flag) {
    ctx->experts_loaded = false;
    return fail(ctx, MOE_ERR_NAN_SCALE, "an E8M0 scale byte is 0xFF (NaN)");
  }
  ctx->experts_loaded = true;
  return rc;
}

int moe_load_experts_affine(moe_ctx* ctx, const uint8_t* experts) {
  if (!ctx) return MOE_ERR_INVALID_ARG;
  if (!experts) return fail(ctx, MOE_ERR_INVALID_ARG, "experts is NULL");
  const int bits = ctx->base.aff_bits;
  if (!bits) return fail(ctx, MOE_ERR_INVALID_ARG, "the context holds MXFP4 experts: load them with moe_load_experts");
  DeviceGuard guard(ctx->device);
  const int d = ctx->cfg.d, F = ctx->cfg.ffn;
  const int E = ctx->base.e_end - ctx->base.e_begin;
  const int S = ctx->base.e_begin == 0 ? ctx->cfg.shared_ffn : 0;
  const size_t cs = moe::aff_expert_bytes(d, F, bits);  // canonical bytes per routed expert (= repacked bytes)
  const size_t cs_s = S > 0 ? moe::aff_expert_bytes(d, S, bits) : 0;
  const int per_chunk = (int)std::max<size_t>(1, ((size_t)256 << 20) / cs);
  uint8_t* st = nullptr;
  cudaError_t e = cudaMalloc(&st, std::max(cs * (size_t)std::min(per_chunk, std::max(E, 1)), cs_s));
  if (e != cudaSuccess) return fail(ctx, MOE_ERR_NOMEM, std::string("staging cudaMalloc: ") + cudaGetErrorString(e));
  e = cudaMemset(ctx->load_err, 0, 4);
  for (int x0 = 0; x0 < E && e == cudaSuccess; x0 += per_chunk) {
    const int n = std::min(per_chunk, E - x0);
    if ((e = cudaMemcpy(st, experts + (size_t)x0 * cs, cs * n, cudaMemcpyDefault)) != cudaSuccess) break;
    if ((e = moe::launch_repack_affine(st, n, d, F, bits, cs, ctx->packed + (size_t)x0 * ctx->expert_stride,
                                       ctx->expert_stride, ctx->load_err, 0)) != cudaSuccess)
      break;
    e = cudaDeviceSynchronize();
  }
  if (e == cudaSuccess && S > 0 &&
      (e = cudaMemcpy(st, experts + (size_t)E * cs, cs_s, cudaMemcpyDefault)) == cudaSuccess &&
      (e = moe::launch_repack_affine(st, 1, d, S, bits, cs_s, ctx->packed + (size_t)E * ctx->expert_stride, cs_s,
                                     ctx->load_err, 0)) == cudaSuccess)
    e = cudaDeviceSynchronize();
  int bad = 0;
  if (e == cudaSuccess) e = cudaMemcpy(&bad, ctx->load_err, 4, cudaMemcpyDeviceToHost);
  cudaFree(st);
  if (e != cudaSuccess) return cuda_fail(ctx, e, "affine expert load");
  if (bad) {
    ctx->experts_loaded = false;
    return fail(ctx, MOE_ERR_NAN_SCALE, "an affine scale or bias is Inf or NaN");
  }
  ctx->experts_loaded = true;
  return MOE_OK;
}

int moe_forward(moe_ctx* ctx, const void* x, int T, void* out, void* stream) {
  if (!ctx) return MOE_ERR_INVALID_ARG;
  if (T < 0) return fail(ctx, MOE_ERR_INVALID_ARG, "T < 0");
  if (T > ctx->cfg.t_max) return fail(ctx, MOE_ERR_T_TOO_LARGE, "T exceeds t_max");
  if (!ctx->router_loaded || !ctx->experts_loaded) return fail(ctx, MOE_ERR_NOT_LOADED, "router or experts not loaded");
  if (T > 0 && (!x || !out)) return fail(ctx, MOE_ERR_INVALID_ARG, "x or out is NULL");
  if (T > 0 && (!aligned16(x) || !aligned16(out)))
    return fail(ctx, MOE_ERR_INVALID_ARG, "x and out must be 16-byte aligned");
  DeviceGuard guard(ctx->device);
  moe::FwdParams p = ctx->base;
  p.T = T;
  p.P = T * ctx->cfg.top_k;
  p.x = static_cast<const uint16_t*>(x);
  p.out = out;
  p.bias = ctx->has_bias ? ctx->bias : nullptr;
  p.w_sg = ctx->has_sg ? ctx->w_sg : nullptr;
  ctx->last_T = T;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  cudaError_t e = cudaSuccess;
  if (uses_decode(ctx, T)) {
    moe::DecParams dp = ctx->dec;
    dp.f = p;
    const bool prof = ctx->n_prof >= 2;
    if (prof) cudaEventRecord(ctx->prof[0], s);
    if (ctx->fused_tc_ok) {
      moe::TcLayerParams tp = ctx->tcl;
      tp.d.f = p;
      e = moe::launch_tc_layer(tp, s, ctx->num_sms);
    } else {
      e = moe::launch_decode(dp, s, ctx->num_sms, ctx->max_smem);
    }
    if (prof && e == cudaSuccess) cudaEventRecord(ctx->prof[1], s);
  } else {
    e = moe::launch_forward(p, s, ctx->num_sms, ctx->n_prof == moe::forward_phases(p) + 1 ? ctx->prof : nullptr);
  }
  if (e != cudaSuccess) return cuda_fail(ctx, e, "forward launch");
  return MOE_OK;
}

int moe_forward_host(moe_ctx* ctx, const void* x_host, int T, void* out_host, void* stream, int synchronize) {
  if (!ctx) return MOE_ERR_INVALID_ARG;
  if (T < 0 || T > ctx->cfg.t_max) return moe_forward(ctx, x_host, T, out_host, stream);
  if (T > 0 && (!x_host || !out_host)) return fail(ctx, MOE_ERR_INVALID_ARG, "x or out is NULL");
  DeviceGuard guard(ctx->device);
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const size_t xb = (size_t)T * ctx->cfg.d * 2;
  const size_t ob = (size_t)T * ctx->cfg.d * (ctx->cfg.out_dtype == MOE_OUT_F32 ? 4 : 2);
  cudaError_t e = cudaSuccess;
  // In-place host buffers. A page-locked buffer mapped into the device's
  // address space (cudaHostAlloc / cudaMallocHost, torch pin_memory) is passed
  // to the kernels as is instead of going through the context's staging
  // buffers: no copy-engine operation then sits between consecutive layer
  // kernels on the stream, so each next kernel is still scheduled while the
  // previous one drains (programmatic dependent launch), as with device
  // buffers.
  //  * out: whenever it is mapped. Every kernel that writes y writes each
  //    element once and reads none back, so the link carries y once.
  //  * x: only for the single-launch kernels on at most kMappedXBytes of x.
  //    Every CTA of those kernels stages all of x, so the link carries one
  //    copy of x per SM: measured on GB300, a 5,760-byte token (d = 2880) went
  //    from 36.3 to 28.4 us per layer end to end with both buffers in place,
  //    while 8 tokens of d = 2048 (32 KB) and 16 of d = 2880 (92 KB) were
  //    slower than through the copy. When x and out share bytes, x is copied.
  constexpr size_t kMappedXBytes = 16384;
  const void* od = T > 0 ? mapped_host_address(out_host) : nullptr;
  if (od && !aligned16(od)) od = nullptr;
  const void* xd =
      (T > 0 && xb <= kMappedXBytes && uses_decode(ctx, T)) ? mapped_host_address(x_host) : nullptr;
  if (xd && !aligned16(xd)) xd = nullptr;
  if (xd && od) {
    const uintptr_t x0 = reinterpret_cast<uintptr_t>(x_host), o0 = reinterpret_cast<uintptr_t>(out_host);
    if (!(x0 + xb <= o0 || o0 + ob <= x0)) xd = nullptr;  // y would overwrite x while CTAs still read it
  }
  if (T > 0 && !xd) e = cudaMemcpyAsync(ctx->x_dev, x_host, xb, cudaMemcpyDefault, s);
  if (e != cudaSuccess) return cuda_fail(ctx, e, "x copy");
  int rc = moe_forward(ctx, xd ? xd : ctx->x_dev, T, od ? const_cast<void*>(od) : ctx->out_dev, stream);
  if (rc != MOE_OK) return rc;
  if (T > 0 && !od) e = cudaMemcpyAsync(out_host, ctx->out_dev, ob, cudaMemcpyDefault, s);
  if (e == cudaSuccess && synchronize) e = cudaStreamSynchronize(s);
  if (e != cudaSuccess) return cuda_fail(ctx, e, "out copy");
  return MOE_OK;
}

int moe_get_routing(moe_ctx* ctx, int32_t* ids, float* gates, int32_t* counts, int32_t* offsets, int32_t* perm,
                    int32_t* inv, void* stream) {
  if (!ctx) return MOE_ERR_INVALID_ARG;
  DeviceGuard guard(ctx->device);
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const size_t P = (size_t)ctx->last_T * ctx->cfg.top_k;
  const moe::FwdParams& p = ctx->base;
  cudaError_t e = cudaSuccess;
  if (ids && P && e == cudaSuccess) e = cudaMemcpyAsync(ids, p.ids, P * 4, cudaMemcpyDefault, s);
  if (gates && P && e == cudaSuccess) e = cudaMemcpyAsync(gates, p.gates, P * 4, cudaMemcpyDefault, s);
  if (counts && e == cudaSuccess) e = cudaMemcpyAsync(counts, p.counts, (size_t)ctx->cfg.n_experts * 4, cudaMemcpyDefault, s);
  if (offsets && e == cudaSuccess)
    e = cudaMemcpyAsync(offsets, p.offsets, (size_t)(ctx->cfg.n_experts + 1) * 4, cudaMemcpyDefault, s);
  if (perm && P && e == cudaSuccess) e = cudaMemcpyAsync(perm, p.perm, P * 4, cudaMemcpyDefault, s);
  if (inv && P && e == cudaSuccess) e = cudaMemcpyAsync(inv, p.inv, P * 4, cudaMemcpyDefault, s);
  if (e != cudaSuccess) return cuda_fail(ctx, e, "routing copy");
  return MOE_OK;
}

int moe_get_logits(moe_ctx* ctx, float* hi, float* lo, void* stream) {
  if (!ctx) return MOE_ERR_INVALID_ARG;
  DeviceGuard guard(ctx->device);
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const size_t n = (size_t)ctx->last_T * ctx->cfg.n_experts * 4;
  cudaError_t e = cudaSuccess;
  if (hi && n) e = cudaMemcpyAsync(hi, ctx->base.logit_hi, n, cudaMemcpyDefault, s);
  if (lo && n && e == cudaSuccess) e = cudaMemcpyAsync(lo, ctx->base.logit_lo, n, cudaMemcpyDefault, s);
  if (e != cudaSuccess) return cuda_fail(ctx, e, "logits copy");
  return MOE_OK;
}

int moe_get_status(moe_ctx* ctx, int clear) {
  if (!ctx) return MOE_ERR_INVALID_ARG;
  DeviceGuard guard(ctx->device);
  cudaError_t e = cudaDeviceSynchronize();
  int st = 0;
  if (e == cudaSuccess) e = cudaMemcpy(&st, ctx->base.status, 4, cudaMemcpyDeviceToHost);
  if (e == cudaSuccess && clear) e = cudaMemset(ctx->base.status, 0, 4);
  if (e != cudaSuccess) return cuda_fail(ctx, e, "status read");
  return st;
}


int moe_profile_events(moe_ctx* ctx, void* const* events, int n_events) {
  if (!ctx) return MOE_ERR_INVALID_ARG;
  if (!events || n_events == 0) {
    ctx->n_prof = 0;
    return MOE_OK;
  }
  if (n_events != 2 && n_events != moe::forward_phases(ctx->base) + 1)
    return fail(ctx, MOE_ERR_INVALID_ARG, "n_events must be moe_forward_phases(T) + 1");
  for (int i = 0; i < n_events; ++i) {
    if (!events[i]) return fail(ctx, MOE_ERR_INVALID_ARG, "NULL event");
    ctx->prof[i] = static_cast<cudaEvent_t>(events[i]);
  }
  ctx->n_prof = n_events;
  return MOE_OK;
}

int moe_forward_phases(const moe_ctx* ctx, int T, const char** names) {
  if (!ctx) return MOE_ERR_INVALID_ARG;
  if (uses_decode(ctx, T)) {
    if (names) *names = "layer";
    return 1;
  }
  if (names) *names = ctx->base.tc_gateup ? moe::kForwardPhaseNamesTc : moe::kForwardPhaseNames;
  return moe::forward_phases(ctx->base);
}

int moe_launches_per_forward(const moe_ctx* ctx, int T) {
  if (!ctx) return MOE_ERR_INVALID_ARG;
  if (T <= 0) return 0;
  if (uses_decode(ctx, T)) return 1;
  const int n = ctx->base.tc_gateup ? moe::kLaunchesPerForwardTc : moe::kLaunchesPerForward;
  if (T > moe::kRouteDDMaxT) return n;
  // one router launch instead of router + top-k; without the tcgen05 layout it also prepares the f16 x
  return ctx->base.tc_gateup ? n - 1 : n - 2;
}

size_t moe_weight_bytes(const moe_ctx* ctx) {
  return ctx ? ctx->packed_bytes + ctx->tcw_bytes + ctx->tcwd_bytes : 0;
}

const char* moe_last_error(const moe_ctx* ctx) { return ctx ? ctx->err.c_str() : g_create_error.c_str(); }

void moe_destroy(moe_ctx* ctx) {
  if (!ctx) return;
  {
    DeviceGuard guard(ctx->device);
    cudaFree(ctx->packed);
    cudaFree(ctx->tcw);
    cudaFree(ctx->tcwd);
    cudaFree(ctx->w_router);
    cudaFree(ctx->bias);
    cudaFree(ctx->w_sg);
    cudaFree(ctx->ws);
  }
  delete ctx;
}

}  // extern "C"
