// Gate/up + SwiGLU of the general path on the 5th-generation tensor cores:
// a block-scaled MMA of the MXFP4 expert weights (E2M1 codes with their E8M0
// scales) by MXFP8 activations (tcgen05.mma kind::mxf8f6f4.block_scale),
// accumulators in tensor memory.
//
// The activation x (bf16) enters as two MXFP8 planes, x = 2^sh * hi + 2^sl * lo
// per 32-element block (E4M3 codes hi and lo with their own E8M0 scales): a
// bf16 value has 8 significant bits, hi keeps its top 4 and lo the remaining 4,
// so the split is exact except for elements below about 2^-10 of their block's
// largest one. Token m of a unit is B row m (hi) and B row npad + m (lo); its
// gate (up) value is D[., m] + D[., npad + m].
//
// Work unit: (slot, M tile of 4 pair tiles = 64 gate + 64 up rows, block of
// up to 48 tokens of the slot); K = d in steps of 128 (four K=32 MMAs). The
// weights come from their own copy, one contiguous block per (M tile, K step)
// already in the operand's core-matrix order, and the activations from
// per-(slot, token block) panels packed once per call in the same order, so a
// stage is three bulk copies (cp.async.bulk) issued by one thread. The CTA is
// warp-specialized: a producer lane, four converter warps that widen the
// packed E2M1 codes (8 bytes -> 16 bytes, the MMA's E2M1 operand layout) and
// store the stage's scale factors to tensor memory, an MMA lane, and four
// epilogue warps that read a finished unit's accumulators (double-buffered in
// tensor memory, so the next unit's MMAs run meanwhile) and write h =
// SiLU(gate) * up in the f16 hi + lo format of the down step. Stages are
// handed on with mbarriers: full (bulk bytes landed), ready (operands
// widened, scales stored), empty (the stage's MMAs completed).
//
// The pages: tokens grouped by expert on the GPU for the prompt, one GEMM per
// expert over its rows ("Neural Server" technical page, "Prompt processing").
#include <stdint.h>

#include "../../include/moe.h"
#include "moe_device.cuh"
#include "moe_internal.h"
#include "moe_tc.cuh"

namespace moe {
namespace {

using namespace dev;

constexpr int kThr = 384;                  // 12 warps: see the roles below
constexpr int kStages = 6;                 // bulk-copy stages in flight
constexpr int kMaxTok = kTcGemmRows;       // tokens per unit
constexpr int kStageBytes = kTcBlockBytes + kTcPanelStep;  // [A codes | SFA | B | SFB]
constexpr int kAExp = 128 * kTcStepK;      // widened E2M1 operand: 16 bytes per 16 elements
constexpr uint32_t kTmemCols = 512;        // D: 2 x 128 columns; scale-factor sets from column 256
constexpr int kSfCol = 256;                // set (step & 1): SFA columns +16 set .. +3, SFB +8 .. +11
constexpr long long kWaitNs = 50000000LL;
// roles
constexpr int kProducerWarp = 0, kMmaWarp = 1, kConvWarp0 = 4, kEpiWarp0 = 8;

__device__ __forceinline__ void bounded_wait(uint64_t* bar, uint32_t parity, int* status) {
  if (mbar_try_wait(bar, parity)) return;
  const uint64_t t0 = globaltimer();
  while (!mbar_try_wait(bar, parity)) {
    if ((long long)(globaltimer() - t0) > kWaitNs) {
      atomicCAS(status, 0, MOE_ERR_TIMEOUT);
      return;
    }
  }
}

__device__ __forceinline__ int find_unit_slot(const int32_t* prefix, int n, int unit) {
  int lo = 0, hi = n - 1;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (prefix[mid] <= unit) lo = mid;
    else hi = mid - 1;
  }
  return lo;
}

struct TcUnit {
  int e, f;     // expert (E = shared) and its ffn
  int q0, n;    // first h row and tokens of the block
  int tau0;     // first pair tile
  int panel;    // activation panel of the (slot, token block)
};

__device__ __forceinline__ TcUnit tc_unit(const FwdParams& p, int u) {
  const int ns = *p.n_slots;
  const int s = find_unit_slot(p.gu_prefix, ns, u);
  const int r = u - p.gu_prefix[s];
  TcUnit g;
  g.e = p.slot_expert[s];
  g.f = (g.e == p.E) ? p.S : p.F;
  const int ngrp = tc_msteps(g.f);
  const int tb = r / ngrp, grp = r - tb * ngrp;
  g.q0 = p.slot_q0[s] + kMaxTok * tb;
  g.n = min(kMaxTok, p.slot_n[s] - kMaxTok * tb);
  g.tau0 = 4 * grp;
  g.panel = p.panel_prefix[s] + tb;
  return g;
}

__device__ __forceinline__ int tok_of(const FwdParams& p, int q) { return q < p.P ? p.perm[q] / p.k : q - p.P; }
__device__ __forceinline__ int npad_of(int n) { return max(8, (n + 7) & ~7); }

__global__ void __launch_bounds__(kThr, 1) gemm_gateup_tc_kernel(FwdParams p) {
  extern __shared__ __align__(1024) uint8_t sm[];
  uint8_t* stages = sm;
  uint8_t* aexp = sm + (size_t)kStages * kStageBytes;           // 2 widened A operands
  float* upx = reinterpret_cast<float*>(aexp + 2 * kAExp);      // [64 rows][kMaxTok]
  uint64_t* full = reinterpret_cast<uint64_t*>(upx + 64 * kMaxTok);
  uint64_t* ready = full + kStages;
  uint64_t* empty = ready + kStages;
  uint64_t* accfull = empty + kStages;
  uint64_t* accempty = accfull + 2;
  uint32_t* tslot = reinterpret_cast<uint32_t*>(accempty + 2);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int total = p.gu_prefix[*p.n_slots];
  const int n_units = total > (int)blockIdx.x ? (total - (int)blockIdx.x + gridDim.x - 1) / gridDim.x : 0;
  if (n_units == 0) return;
  // the padding half of every widened 16-byte row chunk stays zero
  for (int o = tid; o < 2 * kAExp / 16; o += kThr) reinterpret_cast<uint4*>(aexp)[o] = make_uint4(0, 0, 0, 0);
  tc::fence_proxy_async();  // visible to the tensor core's reads
  if (tid == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&ready[s], 128);
      mbar_init(&empty[s], 1);
    }
    for (int a = 0; a < 2; ++a) {
      mbar_init(&accfull[a], 1);
      mbar_init(&accempty[a], 128);
    }
    fence_mbar_init();
  }
  if (warp == 0) tc::alloc(tslot, kTmemCols);
  tc::fence_before();
  __syncthreads();
  tc::fence_after();
  const uint32_t tmem = *tslot;
  const int nks = tc_ksteps(p.d);
  const int G = gridDim.x, b0 = blockIdx.x;

  if (warp == kProducerWarp) {
    if (lane == 0) {
      int j = 0;
      for (int i = 0; i < n_units; ++i) {
        const TcUnit g = tc_unit(p, b0 + i * G);
        const int N = 2 * npad_of(g.n);
        const uint8_t* wsrc = p.tcw + (size_t)g.e * p.tcw_stride + (size_t)(g.tau0 / 4) * nks * kTcBlockBytes;
        const uint8_t* psrc = p.xpanel + (size_t)g.panel * nks * kTcPanelStep;
        for (int ks = 0; ks < nks; ++ks, ++j) {
          const int s = j % kStages;
          if (j >= kStages) bounded_wait(&empty[s], (uint32_t)((j / kStages - 1) & 1), p.status);
          uint8_t* sb = stages + (size_t)s * kStageBytes;
          mbar_arrive_expect_tx(&full[s], (uint32_t)(kTcBlockBytes + N * kTcStepK + 512));
          bulk_g2s(sb, wsrc + (size_t)ks * kTcBlockBytes, kTcBlockBytes, &full[s]);
          bulk_g2s(sb + kTcBlockBytes, psrc + (size_t)ks * kTcPanelStep, (uint32_t)(N * kTcStepK), &full[s]);
          bulk_g2s(sb + kTcBlockBytes + kTcPanelRows * kTcStepK, psrc + (size_t)ks * kTcPanelStep + kTcPanelRows * kTcStepK,
                   512, &full[s]);
        }
      }
    }
  } else if (warp >= kConvWarp0 && warp < kConvWarp0 + 4) {
    const int ct = tid - kConvWarp0 * 32, q = warp & 3;
    int j = 0;
    for (int i = 0; i < n_units; ++i) {
      for (int ks = 0; ks < nks; ++ks, ++j) {
        const int s = j % kStages;
        bounded_wait(&full[s], (uint32_t)((j / kStages) & 1), p.status);
        // widened buffer and scale set j & 1 were last read by step j - 2's MMAs
        if (j >= 2) bounded_wait(&empty[(j - 2) % kStages], (uint32_t)(((j - 2) / kStages) & 1), p.status);
        const uint8_t* sb = stages + (size_t)s * kStageBytes;
        uint8_t* ab = aexp + (size_t)(j & 1) * kAExp;
#pragma unroll
        for (int r = 0; r < kTcCodeBytes / 16 / 128; ++r) {
          const int o = ct + 128 * r;  // 16 code bytes = two 8-byte row chunks
          const uint4 v = *reinterpret_cast<const uint4*>(sb + 16 * o);
          *reinterpret_cast<uint2*>(ab + 32 * o) = make_uint2(v.x, v.y);
          *reinterpret_cast<uint2*>(ab + 32 * o + 16) = make_uint2(v.z, v.w);
        }
        const uint32_t lanebase = tmem + ((uint32_t)(q * 32) << 16) + kSfCol + 16 * (j & 1);
        const uint4 wa = *reinterpret_cast<const uint4*>(sb + kTcCodeBytes + 16 * lane);
        const uint4 wb = *reinterpret_cast<const uint4*>(sb + kTcBlockBytes + kTcPanelRows * kTcStepK + 16 * lane);
        tc::st4(lanebase, wa.x, wa.y, wa.z, wa.w);
        tc::st4(lanebase + 8, wb.x, wb.y, wb.z, wb.w);
        tc::wait_st();
        tc::fence_proxy_async();
        tc::fence_before();
        mbar_arrive(&ready[s]);
      }
    }
  } else if (warp == kMmaWarp) {
    if (lane == 0) {
      int j = 0;
      for (int i = 0; i < n_units; ++i) {
        const TcUnit g = tc_unit(p, b0 + i * G);
        const int N = 2 * npad_of(g.n), acc = i & 1;
        if (i >= 2) bounded_wait(&accempty[acc], (uint32_t)((i / 2 - 1) & 1), p.status);
        tc::fence_after();
        for (int ks = 0; ks < nks; ++ks, ++j) {
          const int s = j % kStages;
          bounded_wait(&ready[s], (uint32_t)((j / kStages) & 1), p.status);
          tc::fence_after();
          const uint8_t* ab = aexp + (size_t)(j & 1) * kAExp;
          const uint8_t* bb = stages + (size_t)s * kStageBytes + kTcBlockBytes;
          const uint32_t sf = tmem + kSfCol + 16 * (j & 1);
#pragma unroll
          for (int kb = 0; kb < 4; ++kb) {
            const uint64_t ad = tc::smem_desc(ab + 2 * kb * 128, 128, 8 * 128);
            const uint64_t bd = tc::smem_desc(bb + 2 * kb * 128, 128, 8 * 128);
            tc::mma_mxf4_mxf8(tmem + 128 * acc, ad, bd, tc::idesc_mxf4_mxf8(128, N, kb, kb), sf, sf + 8,
                              (ks > 0 || kb > 0) ? 1u : 0u);
          }
          tc::commit(&empty[s]);
        }
        tc::commit(&accfull[acc]);
      }
    }
  } else if (warp >= kEpiWarp0) {
    const int qd = warp & 3;
    const uint32_t trow = tmem + ((uint32_t)(qd * 32) << 16);
    for (int i = 0; i < n_units; ++i) {
      const TcUnit g = tc_unit(p, b0 + i * G);
      const int npad = npad_of(g.n), acc = i & 1;
      bounded_wait(&accfull[acc], (uint32_t)((i / 2) & 1), p.status);
      tc::fence_after();
      const uint32_t dcol = trow + 128 * acc;
      if (qd >= 2) {  // up rows 64 + 32 (qd - 2) + lane -> shared memory
        for (int c0 = 0; c0 < npad; c0 += 16) {
          float hi[16], lo[16];
          tc::ld16(dcol + c0, hi);
          tc::ld16(dcol + npad + c0, lo);
#pragma unroll
          for (int x = 0; x < 16; ++x)
            if (c0 + x < g.n) upx[(32 * (qd - 2) + lane) * kMaxTok + c0 + x] = hi[x] + lo[x];
        }
      }
      named_bar(1, 128);
      if (qd < 2) {  // gate rows 32 qd + lane: pair tile tau0 + 2 qd + lane / 16, row lane % 16
        const int tau = g.tau0 + 2 * qd + (lane >> 4), r = lane & 15;
        const bool valid = tau < g.f / 16;
        for (int c0 = 0; c0 < npad; c0 += 16) {
          float hi[16], lo[16];
          tc::ld16(dcol + c0, hi);
          tc::ld16(dcol + npad + c0, lo);
#pragma unroll
          for (int x = 0; x < 16; ++x) {
            const int m = c0 + x;
            if (m >= g.n) break;  // uniform over the warp
            const float gate = hi[x] + lo[x];
            const float up = upx[(32 * qd + lane) * kMaxTok + m];
            const float h = gate / (1.f + expf(-gate)) * up;
            float mx = fabsf(h);
            for (int o = 1; o < 16; o <<= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
            if (valid) {
              const int qq = g.q0 + m;
              const int sh = f16_headroom_exponent(mx);
              __half* hh = reinterpret_cast<__half*>(p.hbuf) + (size_t)qq * 2 * p.fmax64;
              const int ii = 32 * (tau >> 1) + 8 * (r >> 2) + 4 * (tau & 1) + (r & 3);
              const float v = h * pow2f(sh);
              const __half vh = __float2half_rn(v);
              hh[ii] = vh;
              hh[p.fmax64 + ii] = __float2half_rn(v - __half2float(vh));
              if (r == 0) p.hscale[(size_t)qq * p.hgroups + tau] = pow2f(-sh);
            }
          }
        }
      }
      tc::fence_before();
      named_bar(1, 128);  // the up buffer and this accumulator are free
      mbar_arrive(&accempty[acc]);
    }
  }
  tc::fence_before();
  __syncthreads();
  if (warp == 0) {
    tc::fence_after();
    tc::dealloc(tmem, kTmemCols);
  }
}

// Activation panels: one CTA per (panel, K step). Panel rows n < 2 npad:
// plane n / npad, token m = n % npad of the block (rows past the block's
// tokens are zero, their scales 127).
__global__ void __launch_bounds__(256) pack_panels_kernel(FwdParams p) {
  const int pb = blockIdx.x, ks = blockIdx.y;
  const int ns = *p.n_slots;
  if (pb >= p.panel_prefix[ns]) return;
  const int s = find_unit_slot(p.panel_prefix, ns, pb);
  const int tb = pb - p.panel_prefix[s];
  const int n = min(kMaxTok, p.slot_n[s] - kMaxTok * tb), q0 = p.slot_q0[s] + kMaxTok * tb, npad = npad_of(n);
  const int nks = tc_ksteps(p.d);
  uint8_t* dst = p.xpanel + ((size_t)pb * nks + ks) * kTcPanelStep;
  for (int o = threadIdx.x; o < kTcPanelRows * 8; o += 256) {  // 16-byte chunks (row, kc)
    const int row = o >> 3, kc = o & 7;
    const int plane = row >= npad, m = row - plane * npad, k0 = kTcStepK * ks + 16 * kc;
    uint4 v = make_uint4(0, 0, 0, 0);
    if (row < 2 * npad && m < n && k0 < p.d64)
      v = *reinterpret_cast<const uint4*>(p.xq + ((size_t)tok_of(p, q0 + m) * 2 + plane) * p.d64 + k0);
    *reinterpret_cast<uint4*>(dst + ((row >> 3) * 8 + kc) * 128 + (row & 7) * 16) = v;
  }
  if (threadIdx.x < 128) {  // scale word (lane l, r) for B row 32 r + l
    const int l = threadIdx.x >> 2, r = threadIdx.x & 3, row = 32 * r + l;
    const int plane = row >= npad, m = row - plane * npad;
    uint32_t w = 0x7F7F7F7Fu;
    if (row < 2 * npad && m < n) {
      const uint8_t* sc = p.xqs + ((size_t)tok_of(p, q0 + m) * 2 + plane) * p.xq_spitch;
      w = 0;
      for (int kb = 0; kb < 4; ++kb) {
        const int blk = 4 * ks + kb;
        w |= (uint32_t)(blk < p.xq_spitch ? sc[blk] : 127) << (8 * kb);
      }
    }
    *reinterpret_cast<uint32_t*>(dst + kTcPanelRows * kTcStepK + 16 * l + 4 * r) = w;
  }
}

// The tcgen05 weight copy: one thread per (expert, M tile, K step, M row).
__global__ void repack_tc_kernel(const uint8_t* codes, const uint8_t* scales, int n_exp, int d, int f,
                                 size_t ccs, size_t css, uint8_t* out, size_t out_stride) {
  const int nms = tc_msteps(f), nks = tc_ksteps(d);
  const long long total = (long long)n_exp * nms * nks * 128;
  for (long long gid = (long long)blockIdx.x * blockDim.x + threadIdx.x; gid < total;
       gid += (long long)gridDim.x * blockDim.x) {
    const int m = (int)(gid & 127);
    const long long blk = gid >> 7;
    const int ks = (int)(blk % nks), a = (int)((blk / nks) % nms), x = (int)(blk / ((long long)nks * nms));
    const int t = m >> 4, rho = m & 15, tau = 4 * a + (t & 3), half = t >> 2;
    const bool live = tau < f / 16;
    const int row = half * f + 32 * (tau >> 1) + 8 * (rho >> 2) + 4 * (tau & 1) + (rho & 3);
    uint8_t* dst = out + (size_t)x * out_stride + ((size_t)a * nks + ks) * kTcBlockBytes;
    const uint8_t* cr = codes + (size_t)x * ccs + (size_t)row * (d / 2);
    const uint8_t* sr = scales + (size_t)x * css + (size_t)row * (d / 32);
    for (int kc = 0; kc < 8; ++kc) {
      const int k0 = kTcStepK * ks + 16 * kc;
      uint2 v = make_uint2(0u, 0u);
      if (live && k0 < d) {
        uint8_t b[8];
        for (int i = 0; i < 8; ++i) b[i] = cr[k0 / 2 + i];
        v.x = (uint32_t)b[0] | ((uint32_t)b[1] << 8) | ((uint32_t)b[2] << 16) | ((uint32_t)b[3] << 24);
        v.y = (uint32_t)b[4] | ((uint32_t)b[5] << 8) | ((uint32_t)b[6] << 16) | ((uint32_t)b[7] << 24);
      }
      *reinterpret_cast<uint2*>(dst + ((m >> 3) * 8 + kc) * 64 + (m & 7) * 8) = v;
    }
    uint32_t w = 0;
    for (int kb = 0; kb < 4; ++kb) {
      const int blk32 = 4 * ks + kb;
      const uint32_t sc = (live && 32 * blk32 < d) ? sr[blk32] : 127u;
      w |= sc << (8 * kb);
    }
    *reinterpret_cast<uint32_t*>(dst + kTcCodeBytes + 16 * (m & 31) + 4 * (m >> 5)) = w;
  }
}

// x -> two MXFP8 planes per 32-element block (one warp per token, a lane per block).
__global__ void __launch_bounds__(256) prep_xq_kernel(FwdParams p) {
  const int warp = (blockIdx.x * blockDim.x + threadIdx.x) >> 5, lane = threadIdx.x & 31;
  if (warp >= p.T) return;
  const int t = warp;
  const int nblk = p.d64 / 32;
  for (int b = lane; b < p.xq_spitch; b += 32) {
    uint8_t* qh = p.xq + (size_t)t * 2 * p.d64 + 32 * b;
    uint8_t* ql = qh + p.d64;
    if (b >= nblk) {  // scale padding
      p.xqs[(size_t)t * 2 * p.xq_spitch + b] = 127;
      p.xqs[(size_t)t * 2 * p.xq_spitch + p.xq_spitch + b] = 127;
      continue;
    }
    float v[32];
    float amax = 0.f;
#pragma unroll
    for (int i = 0; i < 32; ++i) {
      const int k = 32 * b + i;
      v[i] = k < p.d ? __uint_as_float((uint32_t)p.x[(size_t)t * p.d + k] << 16) : 0.f;
      amax = fmaxf(amax, fabsf(v[i]));
    }
    // hi plane: scale 2^sh with amax * 2^-sh in [128, 256)
    int sh = amax > 0.f ? (int)((__float_as_uint(amax) >> 23) & 0xFF) - 127 - 7 : 0;
    sh = max(-127, min(127, sh));
    const float ish = __uint_as_float((uint32_t)(127 - sh) << 23), fsh = __uint_as_float((uint32_t)(127 + sh) << 23);
    float rmax = 0.f;
    uint32_t hc[32];
#pragma unroll
    for (int i = 0; i < 32; ++i) {
      hc[i] = tc::e4m3_encode(v[i] * ish);
      v[i] -= tc::e4m3_decode(hc[i]) * fsh;  // exact: the remainder of a bf16 value
      rmax = fmaxf(rmax, fabsf(v[i]));
    }
    int sl = rmax > 0.f ? (int)((__float_as_uint(rmax) >> 23) & 0xFF) - 127 - 7 : 0;
    sl = max(-127, min(127, sl));
    const float isl = __uint_as_float((uint32_t)(127 - sl) << 23);
#pragma unroll
    for (int i = 0; i < 32; i += 4) {
      uint32_t wh = 0, wl = 0;
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        wh |= hc[i + j] << (8 * j);
        wl |= tc::e4m3_encode(v[i + j] * isl) << (8 * j);
      }
      *reinterpret_cast<uint32_t*>(qh + i) = wh;
      *reinterpret_cast<uint32_t*>(ql + i) = wl;
    }
    p.xqs[(size_t)t * 2 * p.xq_spitch + b] = (uint8_t)(sh + 127);
    p.xqs[(size_t)t * 2 * p.xq_spitch + p.xq_spitch + b] = (uint8_t)(sl + 127);
  }
}

constexpr size_t kTcSmem = (size_t)kStages * kStageBytes + 2 * (size_t)kAExp + (size_t)64 * kMaxTok * 4 +
                           8 * (3 * kStages + 4) + 16;

}  // namespace

cudaError_t launch_repack_tc(const uint8_t* codes, const uint8_t* scales, int n_exp, int d, int f,
                             size_t canon_code_stride, size_t canon_scale_stride, uint8_t* out, size_t out_stride,
                             cudaStream_t stream) {
  repack_tc_kernel<<<1024, 256, 0, stream>>>(codes, scales, n_exp, d, f, canon_code_stride, canon_scale_stride, out,
                                             out_stride);
  return cudaGetLastError();
}

cudaError_t launch_gemm_gateup_tc(const FwdParams& p, cudaStream_t stream, int num_sms) {
  static bool configured = false;
  if (!configured) {
    cudaError_t e = cudaFuncSetAttribute(gemm_gateup_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kTcSmem);
    if (e != cudaSuccess) return e;
    configured = true;
  }
  prep_xq_kernel<<<(p.T + 7) / 8, 256, 0, stream>>>(p);
  // panels: at most ceil(Q / 48) + slots blocks (the kernel skips the ones past the count)
  const int max_panels = (p.P + p.T) / kTcGemmRows + p.E + 2;
  pack_panels_kernel<<<dim3(max_panels, tc_ksteps(p.d)), 256, 0, stream>>>(p);
  gemm_gateup_tc_kernel<<<num_sms, kThr, kTcSmem, stream>>>(p);
  return cudaGetLastError();
}

}  // namespace moe
