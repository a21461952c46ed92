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
constexpr int kMaxTok = kTcGemmRows;       // tokens per unit
constexpr int kSA = 8;                     // weight stages in flight (bulk copies from HBM)
constexpr int kAOp = 128 * kTcStepK;       // widened E2M1 operand: 16 bytes per 16 elements
constexpr int kAStage = kAOp + 512;        // [operand (packed codes land in its first half) | SFA]
constexpr uint32_t kTmemCols = 512;        // D: 2 buffers at columns 0 and 192; scale factors from 384
constexpr int kDCol = 192;                 // D buffer stride (N <= 192)
constexpr int kSfCol = 384;                // set s (the weight stage): SFA columns +16 s .. +3, SFB +8 .. +15
constexpr long long kWaitNs = 50000000LL;
// roles
constexpr int kProducerWarp = 0, kMmaWarp = 1, kConvWarp0 = 4, kEpiWarp0 = 8;

// The two uses of the GEMM. Gate/up: M tiles of 64 gate + 64 up rows, K = d,
// B = x in 2 MXFP8 planes, epilogue h = SiLU(gate) * up. Down: M tiles of
// 128 rows of d, K = f, B = h in 4 MXFP8 planes, epilogue part = D.
template <bool kDown>
struct Mode {
  static constexpr int kPlanes = kDown ? 4 : 2;
  static constexpr int kPanelRows = kDown ? kTcPanelRowsD : kTcPanelRows;
  static constexpr int kPanelStep = kDown ? kTcPanelStepD : kTcPanelStep;
  static constexpr int kSfWords = kDown ? 8 : 4;  // B scale words per lane in a panel step
  static constexpr int kSB = kDown ? 3 : 5;       // activation-panel stages (from L2)
};

// Per-slot tables the roles look units up in, copied to shared memory once:
// unit prefix, panel prefix, expert, first row, rows (E + 2 entries each).
constexpr size_t tc_table_bytes(int E) { return (size_t)5 * (E + 2) * 4; }

template <bool kDown>
constexpr size_t tc_smem_fixed() {
  return (size_t)kSA * kAStage + (size_t)Mode<kDown>::kSB * Mode<kDown>::kPanelStep +
         (kDown ? 0 : (size_t)64 * kMaxTok * 4) + 8 * (3 * kSA + 2 * Mode<kDown>::kSB + 4) + 16;
}

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

struct SlotTab {
  const int* upre;   // units before each slot
  const int* ppre;   // panels before each slot
  const int* sexp;   // expert of each slot
  const int* sq0;    // first row of each slot
  const int* sn;     // rows of each slot
  int ns;
};

struct TcUnit {
  int e, f;     // expert (E = shared) and its ffn
  int q0, n;    // first h/part row and tokens of the block
  int mt;       // M tile
  int nks;      // K steps
  int panel;    // panel of the (slot, token block)
  const uint8_t* w;  // weight blocks of the M tile (K step 0)
};

template <bool kDown>
__device__ __forceinline__ TcUnit tc_unit(const FwdParams& p, const SlotTab& st, int u) {
  const int s = find_unit_slot(st.upre, st.ns, u);
  const int r = u - st.upre[s];
  TcUnit g;
  g.e = st.sexp[s];
  g.f = (g.e == p.E) ? p.S : p.F;
  const int ngrp = kDown ? tc_dtiles(p.d) : tc_msteps(g.f);
  const int tb = r / ngrp;
  g.mt = r - tb * ngrp;
  g.q0 = st.sq0[s] + kMaxTok * tb;
  g.n = min(kMaxTok, st.sn[s] - kMaxTok * tb);
  g.nks = tc_ksteps(kDown ? g.f : p.d);
  g.panel = st.ppre[s] + tb;
  g.w = kDown ? p.tcwd + (size_t)g.e * p.tcwd_stride + (size_t)g.mt * g.nks * kTcBlockBytes
              : p.tcw + (size_t)g.e * p.tcw_stride + (size_t)g.mt * g.nks * kTcBlockBytes;
  return g;
}

__device__ __forceinline__ int tok_of(const FwdParams& p, int q) { return q < p.P ? p.perm[q] / p.k : q - p.P; }
__device__ __forceinline__ int npad_of(int n) { return max(8, (n + 7) & ~7); }

// The producer's walk over the steps (unit, K step) of the CTA.
template <bool kDown>
struct Cursor {
  int i, ks;
  TcUnit g;
};

template <bool kDown>
__device__ __forceinline__ void cursor_next(const FwdParams& p, const SlotTab& st, Cursor<kDown>& c, int n_units) {
  if (++c.ks == c.g.nks) {
    c.ks = 0;
    if (++c.i < n_units) c.g = tc_unit<kDown>(p, st, blockIdx.x + c.i * gridDim.x);
  }
}

template <bool kDown>
__global__ void __launch_bounds__(kThr, 1) gemm_tc_kernel(FwdParams p) {
  using M = Mode<kDown>;
  constexpr int kSB = M::kSB;
  extern __shared__ __align__(1024) uint8_t sm[];
  uint8_t* astg = sm;                                              // [kSA][kAStage]
  uint8_t* bstg = astg + (size_t)kSA * kAStage;                   // [kSB][panel step]
  float* upx = reinterpret_cast<float*>(bstg + (size_t)kSB * M::kPanelStep);  // gate/up: [64 rows][kMaxTok]
  uint64_t* bars = reinterpret_cast<uint64_t*>(reinterpret_cast<uint8_t*>(upx) + (kDown ? 0 : 64 * kMaxTok * 4));
  uint64_t* fullA = bars;                 // bulk weight bytes landed
  uint64_t* emptyA = fullA + kSA;         // the MMAs reading the weight stage completed
  uint64_t* ready = emptyA + kSA;         // the stage's operand is widened and its scale set stored
  uint64_t* fullB = ready + kSA;          // bulk panel bytes landed
  uint64_t* emptyB = fullB + kSB;         // the MMAs reading the panel stage completed
  uint64_t* accfull = emptyB + kSB;       // [2]
  uint64_t* accempty = accfull + 2;       // [2]
  uint32_t* tslot = reinterpret_cast<uint32_t*>(accempty + 2);
  int* tab = reinterpret_cast<int*>(tslot + 4);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int ns = *p.n_slots;
  const int total = (kDown ? p.dn_prefix : p.gu_prefix)[ns];
  const int n_units = total > (int)blockIdx.x ? (total - (int)blockIdx.x + gridDim.x - 1) / gridDim.x : 0;
  if (n_units == 0) return;
  SlotTab st;
  st.ns = ns;
  st.upre = tab;
  st.ppre = tab + (p.E + 2);
  st.sexp = tab + 2 * (p.E + 2);
  st.sq0 = tab + 3 * (p.E + 2);
  st.sn = tab + 4 * (p.E + 2);
  for (int i = tid; i <= ns; i += kThr) {
    tab[i] = (kDown ? p.dn_prefix : p.gu_prefix)[i];
    tab[(p.E + 2) + i] = p.panel_prefix[i];
    if (i < ns) {
      tab[2 * (p.E + 2) + i] = p.slot_expert[i];
      tab[3 * (p.E + 2) + i] = p.slot_q0[i];
      tab[4 * (p.E + 2) + i] = p.slot_n[i];
    }
  }
  if (tid == 0) {
    for (int s = 0; s < kSA; ++s) {
      mbar_init(&fullA[s], 1);
      mbar_init(&emptyA[s], 1);
      mbar_init(&ready[s], 128);
    }
    for (int s = 0; s < kSB; ++s) {
      mbar_init(&fullB[s], 1);
      mbar_init(&emptyB[s], 1);
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
  const int G = gridDim.x, b0 = blockIdx.x;

  if (warp == kProducerWarp) {
    if (lane == 0) {
      // weights run kSA - kSB steps ahead of the panels: both wait for the
      // same point of the pipeline when their stage comes round
      Cursor<kDown> ca, cb;
      ca.i = cb.i = 0;
      ca.ks = cb.ks = 0;
      ca.g = cb.g = tc_unit<kDown>(p, st, b0);
      int ja = 0, jb = 0;
      while (ca.i < n_units || cb.i < n_units) {
        if (ca.i < n_units && (cb.i >= n_units || ja - jb < kSA - kSB)) {
          const int s = ja % kSA;
          if (ja >= kSA) bounded_wait(&emptyA[s], (uint32_t)((ja / kSA - 1) & 1), p.status);
          uint8_t* sb = astg + (size_t)s * kAStage;
          mbar_arrive_expect_tx(&fullA[s], (uint32_t)kTcBlockBytes);
          bulk_g2s(sb, ca.g.w + (size_t)ca.ks * kTcBlockBytes, kTcCodeBytes, &fullA[s]);
          bulk_g2s(sb + kAOp, ca.g.w + (size_t)ca.ks * kTcBlockBytes + kTcCodeBytes, 512, &fullA[s]);
          ++ja;
          cursor_next<kDown>(p, st, ca, n_units);
        } else {
          const int s = jb % kSB;
          if (jb >= kSB) bounded_wait(&emptyB[s], (uint32_t)((jb / kSB - 1) & 1), p.status);
          const int N = M::kPlanes * npad_of(cb.g.n);
          uint8_t* sb = bstg + (size_t)s * M::kPanelStep;
          // panels of every slot use the stride of the largest K step count
          const int pstride = kDown ? tc_ksteps(p.F > p.S ? p.F : p.S) : tc_ksteps(p.d);
          const uint8_t* src = (kDown ? p.hpanel : p.xpanel) + ((size_t)cb.g.panel * pstride + cb.ks) * M::kPanelStep;
          mbar_arrive_expect_tx(&fullB[s], (uint32_t)(N * kTcStepK + 32 * 4 * M::kSfWords));
          bulk_g2s(sb, src, (uint32_t)(N * kTcStepK), &fullB[s]);
          bulk_g2s(sb + M::kPanelRows * kTcStepK, src + M::kPanelRows * kTcStepK, 32 * 4 * M::kSfWords, &fullB[s]);
          ++jb;
          cursor_next<kDown>(p, st, cb, n_units);
        }
      }
    }
  } else if (warp >= kConvWarp0 && warp < kConvWarp0 + 4) {
    const int ct = tid - kConvWarp0 * 32, q = warp & 3;
    int j = 0;
    for (int i = 0; i < n_units; ++i) {
      const TcUnit g = tc_unit<kDown>(p, st, b0 + i * G);
      for (int ks = 0; ks < g.nks; ++ks, ++j) {
        const int sa = j % kSA, sbi = j % kSB;
        bounded_wait(&fullA[sa], (uint32_t)((j / kSA) & 1), p.status);
        bounded_wait(&fullB[sbi], (uint32_t)((j / kSB) & 1), p.status);
        uint8_t* ap = astg + (size_t)sa * kAStage;
        const uint8_t* sb_p = bstg + (size_t)sbi * M::kPanelStep;
        // widen in place: every converter thread reads its packed chunks, then
        // (after the converters' barrier) writes each 8 bytes into its 16-byte slot
        uint4 v[kTcCodeBytes / 16 / 128];
#pragma unroll
        for (int r = 0; r < kTcCodeBytes / 16 / 128; ++r) v[r] = *reinterpret_cast<const uint4*>(ap + 16 * (ct + 128 * r));
        const uint4 wa = *reinterpret_cast<const uint4*>(ap + kAOp + 16 * lane);
        const uint4 wb0 = *reinterpret_cast<const uint4*>(sb_p + M::kPanelRows * kTcStepK + 4 * M::kSfWords * lane);
        uint4 wb1 = make_uint4(0, 0, 0, 0);
        if (kDown) wb1 = *reinterpret_cast<const uint4*>(sb_p + M::kPanelRows * kTcStepK + 4 * M::kSfWords * lane + 16);
        named_bar(2, 128);
#pragma unroll
        for (int r = 0; r < kTcCodeBytes / 16 / 128; ++r) {
          const int o = ct + 128 * r;  // 16 code bytes = two 8-byte row chunks
          *reinterpret_cast<uint4*>(ap + 32 * o) = make_uint4(v[r].x, v[r].y, 0u, 0u);
          *reinterpret_cast<uint4*>(ap + 32 * o + 16) = make_uint4(v[r].z, v[r].w, 0u, 0u);
        }
        // scale set sa: free, the MMAs of the stage's previous step completed before it was refilled
        const uint32_t lanebase = tmem + ((uint32_t)(q * 32) << 16) + kSfCol + 16 * sa;
        tc::st4(lanebase, wa.x, wa.y, wa.z, wa.w);
        tc::st4(lanebase + 8, wb0.x, wb0.y, wb0.z, wb0.w);
        if (kDown) tc::st4(lanebase + 12, wb1.x, wb1.y, wb1.z, wb1.w);
        tc::wait_st();
        tc::fence_proxy_async();
        tc::fence_before();
        mbar_arrive(&ready[sa]);
      }
    }
  } else if (warp == kMmaWarp) {
    if (lane == 0) {
      int j = 0;
      for (int i = 0; i < n_units; ++i) {
        const TcUnit g = tc_unit<kDown>(p, st, b0 + i * G);
        const int N = M::kPlanes * npad_of(g.n), acc = i & 1;
        if (i >= 2) bounded_wait(&accempty[acc], (uint32_t)((i / 2 - 1) & 1), p.status);
        tc::fence_after();
        for (int ks = 0; ks < g.nks; ++ks, ++j) {
          const int sa = j % kSA;
          bounded_wait(&ready[sa], (uint32_t)((j / kSA) & 1), p.status);
          tc::fence_after();
          const uint8_t* ab = astg + (size_t)sa * kAStage;
          const uint8_t* bb = bstg + (size_t)(j % kSB) * M::kPanelStep;
          const uint32_t sf = tmem + kSfCol + 16 * sa;
#pragma unroll
          for (int kb = 0; kb < 4; ++kb) {
            const uint64_t ad = tc::smem_desc(ab + 2 * kb * 128, 128, 8 * 128);
            const uint64_t bd = tc::smem_desc(bb + 2 * kb * 128, 128, 8 * 128);
            tc::mma_mxf4_mxf8(tmem + kDCol * acc, ad, bd, tc::idesc_mxf4_mxf8(128, N, kb, kb), sf, sf + 8,
                              (ks > 0 || kb > 0) ? 1u : 0u);
          }
          tc::commit(&emptyA[sa]);
          tc::commit(&emptyB[j % kSB]);
        }
        tc::commit(&accfull[acc]);
      }
    }
  } else if (warp >= kEpiWarp0) {
    const int qd = warp & 3;
    const uint32_t trow = tmem + ((uint32_t)(qd * 32) << 16);
    for (int i = 0; i < n_units; ++i) {
      const TcUnit g = tc_unit<kDown>(p, st, b0 + i * G);
      const int npad = npad_of(g.n), acc = i & 1;
      bounded_wait(&accfull[acc], (uint32_t)((i / 2) & 1), p.status);
      tc::fence_after();
      const uint32_t dcol = trow + kDCol * acc;
      if (kDown) {  // part rows q0 + m, column 128 mt + 32 qd + lane: the sum of the 4 planes
        const int row = 128 * g.mt + 32 * qd + lane;
        for (int c0 = 0; c0 < npad; c0 += 16) {
          float v[16], w[16];
          tc::ld16(dcol + c0, v);
#pragma unroll
          for (int pl = 1; pl < 4; ++pl) {
            tc::ld16(dcol + pl * npad + c0, w);
#pragma unroll
            for (int x = 0; x < 16; ++x) v[x] += w[x];
          }
          if (row < p.d) {
#pragma unroll
            for (int x = 0; x < 16; ++x)
              if (c0 + x < g.n) p.part[(size_t)(g.q0 + c0 + x) * p.d + row] = v[x];
          }
        }
      } else {
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
        if (qd < 2) {  // gate rows 32 qd + lane: pair tile 4 mt + 2 qd + lane / 16, row lane % 16
          const int tau = 4 * g.mt + 2 * qd + (lane >> 4), r = lane & 15;
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

// Split the 32 values of a block (one per lane) into `planes` MXFP8 planes:
// each an E8M0 block scale (largest magnitude into [128, 256)) and E4M3 codes
// of what the planes before left over. Plane pl's code goes to code[pl], its
// scale byte is returned in the matching entry of sc (the same in every lane).
template <int kPl>
__device__ __forceinline__ void split_planes(float v, uint32_t (&code)[kPl], uint32_t (&sc)[kPl]) {
#pragma unroll
  for (int pl = 0; pl < kPl; ++pl) {
    float amax = fabsf(v);
    for (int o = 16; o; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
    int sh = amax > 0.f ? (int)((__float_as_uint(amax) >> 23) & 0xFF) - 127 - 7 : 0;
    sh = max(-127, min(127, sh));
    const float ish = __uint_as_float((uint32_t)(127 - sh) << 23), fsh = __uint_as_float((uint32_t)(127 + sh) << 23);
    // E4M3 by the hardware conversions (round to nearest even, saturating at 448)
    uint16_t c2;
    asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(c2) : "f"(0.f), "f"(v * ish));
    uint32_t h2;
    asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(h2) : "h"(c2));
    code[pl] = c2 & 0xFFu;
    v -= __half2float(__ushort_as_half((unsigned short)(h2 & 0xFFFFu))) * fsh;  // the remainder for the next plane
    sc[pl] = (uint32_t)(sh + 127);
  }
}

// h panels of the down step: one CTA per (panel, K step over f), a warp per
// (token row m, 32-element block b of the step), a lane per element. h comes
// from its f16 hi + lo planes and their per-pair-tile scale.
__global__ void __launch_bounds__(256) pack_h_panels_kernel(FwdParams p) {
  const int pb = blockIdx.x, ks = blockIdx.y;
  const int ns = *p.n_slots;
  if (pb >= p.panel_prefix[ns]) return;
  const int s = find_unit_slot(p.panel_prefix, ns, pb);
  const int tb = pb - p.panel_prefix[s];
  const int f = (p.slot_expert[s] == p.E) ? p.S : p.F, nks = tc_ksteps(f);
  if (ks >= nks) return;
  const int n = min(kMaxTok, p.slot_n[s] - kMaxTok * tb), q0 = p.slot_q0[s] + kMaxTok * tb, npad = npad_of(n);
  uint8_t* dst = p.hpanel + ((size_t)pb * tc_ksteps(p.F > p.S ? p.F : p.S) + ks) * kTcPanelStepD;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  for (int o = warp; o < npad * 4; o += 8) {
    const int m = o >> 2, b = o & 3, k = kTcStepK * ks + 32 * b + lane;
    float h = 0.f;
    if (m < n && k < f) {
      const int q = q0 + m;
      const __half* hh = reinterpret_cast<const __half*>(p.hbuf) + (size_t)q * 2 * p.fmax64;
      // the scale of h is per pair tile: element k belongs to pair tile 2 (k / 32) + (k / 4) % 2
      h = (__half2float(hh[k]) + __half2float(hh[p.fmax64 + k])) *
          p.hscale[(size_t)q * p.hgroups + 2 * (k >> 5) + ((k >> 2) & 1)];
    }
    uint32_t code[4], sc[4];
    split_planes<4>(h, code, sc);
#pragma unroll
    for (int pl = 0; pl < 4; ++pl) {
      const int row = pl * npad + m;
      dst[((row >> 3) * 8 + 2 * b + (lane >> 4)) * 128 + (row & 7) * 16 + (lane & 15)] = (uint8_t)code[pl];
      // scale byte b of the word of B row `row`: word (lane row % 32, r row / 32)
      if (lane == 0) dst[kTcPanelRowsD * kTcStepK + 4 * 8 * (row & 31) + 4 * (row >> 5) + b] = (uint8_t)sc[pl];
    }
  }
  // scale bytes of rows past the block's 4 npad rows (the words the MMA reads: r < 8)
  for (int o = threadIdx.x; o < 32 * 8 * 4; o += 256) {
    const int l = o >> 5, r = (o >> 2) & 7, bb = o & 3, row = 32 * r + l;
    if (row >= 4 * npad) dst[kTcPanelRowsD * kTcStepK + 4 * 8 * l + 4 * r + bb] = 127;
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

// The tcgen05 weight copies: one thread per (expert, M tile, K step, M row).
// Gate/up: M row m of tile a is row m % 16 of pair tile 4a + (m / 16) % 4
// (gate rows for m < 64, up rows after), K = d. Down: row 128a + m of the
// down matrix, K = f.
__global__ void repack_tc_kernel(const uint8_t* codes, const uint8_t* scales, int n_exp, int d, int f,
                                 size_t ccs, size_t css, uint8_t* out, size_t out_stride, bool down) {
  const int nms = down ? tc_dtiles(d) : tc_msteps(f), K = down ? f : d, nks = tc_ksteps(K);
  const long long total = (long long)n_exp * nms * nks * 128;
  for (long long gid = (long long)blockIdx.x * blockDim.x + threadIdx.x; gid < total;
       gid += (long long)gridDim.x * blockDim.x) {
    const int m = (int)(gid & 127);
    const long long blk = gid >> 7;
    const int ks = (int)(blk % nks), a = (int)((blk / nks) % nms), x = (int)(blk / ((long long)nks * nms));
    bool live;
    const uint8_t* cr;
    const uint8_t* sr;
    if (down) {
      const int row = 128 * a + m;
      live = row < d;
      cr = codes + (size_t)x * ccs + (size_t)2 * f * d / 2 + (size_t)row * (f / 2);
      sr = scales + (size_t)x * css + (size_t)2 * f * d / 32 + (size_t)row * (f / 32);
    } else {
      const int t = m >> 4, rho = m & 15, tau = 4 * a + (t & 3), half = t >> 2;
      live = tau < f / 16;
      const int row = half * f + 32 * (tau >> 1) + 8 * (rho >> 2) + 4 * (tau & 1) + (rho & 3);
      cr = codes + (size_t)x * ccs + (size_t)row * (d / 2);
      sr = scales + (size_t)x * css + (size_t)row * (d / 32);
    }
    uint8_t* dst = out + (size_t)x * out_stride + ((size_t)a * nks + ks) * kTcBlockBytes;
    for (int kc = 0; kc < 8; ++kc) {
      const int k0 = kTcStepK * ks + 16 * kc;
      uint2 v = make_uint2(0u, 0u);
      if (live && k0 < K) {
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
      const uint32_t sc = (live && 32 * blk32 < K) ? sr[blk32] : 127u;
      w |= sc << (8 * kb);
    }
    *reinterpret_cast<uint32_t*>(dst + kTcCodeBytes + 16 * (m & 31) + 4 * (m >> 5)) = w;
  }
}

// x -> two MXFP8 planes per 32-element block: a warp per (token, block), a lane per element.
__global__ void __launch_bounds__(256) prep_xq_kernel(FwdParams p) {
  const int item = (blockIdx.x * blockDim.x + threadIdx.x) >> 5, lane = threadIdx.x & 31;
  const int nb = p.xq_spitch;  // blocks per row, scale padding included
  if (item >= p.T * nb) return;
  const int t = item / nb, b = item - t * nb;
  uint8_t* qs = p.xqs + (size_t)t * 2 * p.xq_spitch + b;
  if (32 * b >= p.d64) {  // scale padding
    if (lane == 0) {
      qs[0] = 127;
      qs[p.xq_spitch] = 127;
    }
    return;
  }
  const int k = 32 * b + lane;
  const float v = k < p.d ? __uint_as_float((uint32_t)p.x[(size_t)t * p.d + k] << 16) : 0.f;
  uint32_t code[2], sc[2];
  split_planes<2>(v, code, sc);
  uint8_t* qh = p.xq + (size_t)t * 2 * p.d64 + k;
  qh[0] = (uint8_t)code[0];
  qh[p.d64] = (uint8_t)code[1];
  if (lane == 0) {
    qs[0] = (uint8_t)sc[0];
    qs[p.xq_spitch] = (uint8_t)sc[1];
  }
}

}  // namespace

cudaError_t launch_repack_tc(const uint8_t* codes, const uint8_t* scales, int n_exp, int d, int f,
                             size_t canon_code_stride, size_t canon_scale_stride, uint8_t* out, size_t out_stride,
                             bool down, cudaStream_t stream) {
  repack_tc_kernel<<<1024, 256, 0, stream>>>(codes, scales, n_exp, d, f, canon_code_stride, canon_scale_stride, out,
                                             out_stride, down);
  return cudaGetLastError();
}

cudaError_t launch_gemm_gateup_tc(const FwdParams& p, cudaStream_t stream, int num_sms) {
  static bool configured = false;
  if (!configured) {
    cudaError_t e = cudaFuncSetAttribute(gemm_tc_kernel<false>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)(tc_smem_fixed<false>() + tc_table_bytes(512)));
    if (e != cudaSuccess) return e;
    configured = true;
  }
  prep_xq_kernel<<<(p.T * p.xq_spitch + 7) / 8, 256, 0, stream>>>(p);
  // panels: at most ceil(Q / 48) + slots blocks (the kernels skip the ones past the count)
  const int max_panels = (p.P + p.T) / kTcGemmRows + p.E + 2;
  pack_panels_kernel<<<dim3(max_panels, tc_ksteps(p.d)), 256, 0, stream>>>(p);
  gemm_tc_kernel<false><<<num_sms, kThr, tc_smem_fixed<false>() + tc_table_bytes(p.E), stream>>>(p);
  return cudaGetLastError();
}

cudaError_t launch_gemm_down_tc(const FwdParams& p, cudaStream_t stream, int num_sms) {
  static bool configured = false;
  if (!configured) {
    cudaError_t e = cudaFuncSetAttribute(gemm_tc_kernel<true>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)(tc_smem_fixed<true>() + tc_table_bytes(512)));
    if (e != cudaSuccess) return e;
    configured = true;
  }
  const int max_panels = (p.P + p.T) / kTcGemmRows + p.E + 2;
  pack_h_panels_kernel<<<dim3(max_panels, tc_ksteps(p.F > p.S ? p.F : p.S)), 256, 0, stream>>>(p);
  gemm_tc_kernel<true><<<num_sms, kThr, tc_smem_fixed<true>() + tc_table_bytes(p.E), stream>>>(p);
  return cudaGetLastError();
}

}  // namespace moe
