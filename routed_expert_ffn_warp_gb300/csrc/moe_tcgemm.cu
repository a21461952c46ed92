// Gate/up + SwiGLU and the down projection of the general path on the
// 5th-generation tensor cores: block-scaled MMAs of the MXFP4 expert weights
// (E2M1 codes with their E8M0 scales) by MXFP8 activations
// (tcgen05.mma kind::mxf8f6f4.block_scale), accumulators in tensor memory.
//
// The activation x (bf16) enters as two MXFP8 planes, x = 2^sh * hi + 2^sl * lo
// per 32-element block (E4M3 codes hi and lo with their own E8M0 scales): a
// bf16 value has 8 significant bits, hi keeps its top 4 and lo the remaining 4,
// so the split is exact except for elements below about 2^-10 of their block's
// largest one. Token m of a unit is B row m (hi) and B row npad + m (lo); its
// gate (up) value is D[., m] + D[., npad + m]. h enters the down GEMM the same
// way in four planes (about 16 significant bits per block).
//
// Work unit: (slot, pair of M tiles, block of up to 48 tokens of the slot), K
// in steps of 128 (four K=32 MMAs per M tile). Gate/up: M tile = 64 gate + 64
// up rows (4 pair tiles), K = d. Down: M tile = 128 rows of d, K = f. The two
// M tiles of a unit share each K step's activation panel. The weights come from
// their own copy, one contiguous block per (M tile, K step) in the operand's
// core-matrix order with the E2M1 codes packed; a TMA tensor copy of the
// 4-bit "16 x U4, 16-byte aligned" type widens every 8 code bytes to the
// 16-byte rows the MMA reads on the way into shared memory. The activations
// come from per-(slot, token block) panels in the MMA's order: x panels are
// packed once per call, h panels are written by the gate/up epilogue itself.
//
// The CTA is warp-specialized: a weight producer lane (tensor copies, and L2
// prefetches further ahead), an activation producer lane (bulk copies), MMA
// lanes that take the K steps in turn, four warps that move each stage's
// scale factors to tensor memory (tcgen05.st, one per lane quadrant), and
// eight epilogue warps that read a finished unit's accumulators. Stages are
// handed on with mbarriers: full (bytes landed), ready (scale factors in
// tensor memory), empty (the stage's MMAs completed), accfull / accempty
// (accumulator states).
//
// The pages: tokens grouped by expert on the GPU for the prompt, one GEMM per
// expert over its rows ("Neural Server" technical page, "Prompt processing").
#include <cuda.h>
#include <cudaTypedefs.h>
#include <stdint.h>

#include "../../include/moe.h"
#include "moe_device.cuh"
#include "moe_internal.h"
#include "moe_tc.cuh"

namespace moe {
namespace {

using namespace dev;

constexpr int kThr = 512;                  // 16 warps: see the roles below
constexpr int kMaxTok = kTcGemmRows;       // tokens per unit
constexpr int kAOp = 128 * kTcStepK;       // widened E2M1 operand: 16 bytes per 16 elements
constexpr int kCmRows = kTcPairBytes / 64;  // 64-byte tensor rows per weight block of a tile pair
constexpr uint32_t kTmemCols = 512;        // accumulators from column 0, scale factors from 384
constexpr int kSfCol = 384;                // set s (the stage) at +32 s: SFA of M tile 0 / 1 at +0 / +8, SFB at +16
constexpr int kSfSet = 32;
// roles: warp 0 weights, 1 activations, 2 and 3 MMA lanes, 4 .. 7 scale factors to TMEM, 8 .. 15
// epilogue (a warp's TMEM lane quadrant is warp % 4)
constexpr int kProducerWarp = 0, kPanelWarp = 1, kMmaWarp0 = 2, kSfWarp0 = 4, kEpiWarp0 = 8, kEpiThreads = 256;
constexpr int kEpiPerQuad = kEpiThreads / 128;  // epilogue warps per TMEM lane quadrant

// The two uses of the GEMM. Gate/up: M tiles of 64 gate + 64 up rows, K = d,
// B = x in 2 MXFP8 planes, epilogue h = SiLU(gate) * up into the h panels.
// Down: M tiles of 128 rows of d, K = f, B = h in 4 MXFP8 planes, epilogue
// part = D. A stage holds one K step of both operands: [A of M tile 0 | A of
// M tile 1 | SFA of both | B panel step with its SFB]. MMA lane t issues the
// MMAs of M tile t of the unit into its own accumulator.
template <bool kDown>
struct Mode {
  static constexpr int kPlanes = kDown ? 4 : 2;
  static constexpr int kPanelStep = kDown ? kTcPanelStepD : kTcPanelStep;
  static constexpr int kSfBlocks = kDown ? 2 : 1;  // 512-byte B scale blocks per panel step (32 rows x 4 words each)
  static constexpr int kAPair = 2 * kAOp + 1024;
  static constexpr int kStage = kAPair + kPanelStep;
  static constexpr int kS = kDown ? 3 : 4;         // stages
  static constexpr int kMma = 2;                   // MMA lanes = M tiles of a unit
  static constexpr int kDCol = kDown ? 192 : 96;   // accumulator width (N <= kDCol); buffer b, lane t at kDCol (kMma b + t)
  static constexpr int kBufs = kDown ? 1 : 2;      // accumulator buffers (units in flight between MMA and epilogue)
  // L2 prefetch distance of the weight blocks, in K steps. Measured on the
  // 1,024-token prefill layer (us per layer of the GEMM): gate/up 0 / 3 / 4 /
  // 6 / 8 steps 249.7 / 237.7 / 236.1-237.4 / 238.4 / 238.7 (longer windows
  // compete with its panel reads); down 8 / 12 / 24 steps 156.6 / 157.5-159.1 /
  // 203.0.
  static constexpr int kPf = kDown ? 12 : 4;
  static constexpr int kEpiSmem = kDown ? 0 : 4 * kMaxTok * 32 * 4;  // gate/up values of one M tile [4 blocks][token][32]
  static_assert(kBufs * kMma * kDCol <= kSfCol && kSfCol + kS * kSfSet <= (int)kTmemCols, "TMEM columns");
};

// Per-slot tables the roles look units up in, copied to shared memory once:
// unit prefix, panel prefix, expert, first row, rows (E + 2 entries each).
constexpr size_t tc_table_bytes(int E) { return (size_t)5 * (E + 2) * 4; }

template <bool kDown>
constexpr size_t tc_smem_fixed() {
  return (size_t)Mode<kDown>::kS * Mode<kDown>::kStage + Mode<kDown>::kEpiSmem + 8 * (3 * Mode<kDown>::kS + 4) + 16;
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
  int mt, nt;   // first M tile of the pair and tiles in it (1 or 2)
  int nks;      // K steps
  int panel;    // panel of the (slot, token block)
  int y;        // tensor row (64 bytes each) of the pair's first weight block (K step 0)
  const uint8_t* w;  // the pair's weight blocks (K step 0)
};

template <bool kDown>
__device__ __forceinline__ TcUnit tc_unit(const FwdParams& p, const SlotTab& st, int u) {
  const int s = find_unit_slot(st.upre, st.ns, u);
  const int r = u - st.upre[s];
  TcUnit g;
  g.e = st.sexp[s];
  g.f = (g.e == p.E) ? p.S : p.F;
  const int ntiles = kDown ? tc_dtiles(p.d) : tc_msteps(g.f), ngrp = (ntiles + 1) / 2;
  const int tb = r / ngrp;
  g.mt = 2 * (r - tb * ngrp);
  g.nt = min(2, ntiles - g.mt);
  g.q0 = st.sq0[s] + kMaxTok * tb;
  g.n = min(kMaxTok, st.sn[s] - kMaxTok * tb);
  g.nks = tc_ksteps(kDown ? g.f : p.d);
  g.panel = st.ppre[s] + tb;
  const size_t stride = kDown ? p.tcwd_stride : p.tcw_stride;  // a multiple of kTcPairBytes
  const size_t we = (size_t)weight_index(p, g.e);  // the expert's place in this context's copy
  g.y = (int)(we * (stride / 64)) + (g.mt / 2) * g.nks * kCmRows;
  g.w = (kDown ? p.tcwd : p.tcw) + we * stride + (size_t)(g.mt / 2) * g.nks * kTcPairBytes;
  return g;
}

__device__ __forceinline__ int tok_of(const FwdParams& p, int q) { return q < p.P ? p.perm[q] / p.k : q - p.P; }
__device__ __forceinline__ int npad_of(int n) { return max(8, (n + 7) & ~7); }

// Byte offset, within an h panel step of N = 4 npad rows, of the E8M0 scale of
// B row `row` and K block kb: behind the rows, two 512-byte blocks of words
// [lane][4], block r / 4 holding B rows 32 r + lane in word r % 4
// (r = row / 32), the order tcgen05.st writes them to tensor memory.
__device__ __forceinline__ int hsf_off(int npad, int row, int kb) {
  const int r = row >> 5;
  return 4 * npad * kTcStepK + 512 * (r >> 2) + 16 * (row & 31) + 4 * (r & 3) + kb;
}

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
__global__ void __launch_bounds__(kThr, 1) gemm_tc_kernel(const FwdParams p, const __grid_constant__ CUtensorMap wmap) {
  pdl_enter();
  using M = Mode<kDown>;
  constexpr int kS = M::kS, kMma = M::kMma, kBufs = M::kBufs;
  extern __shared__ __align__(1024) uint8_t sm[];
  uint8_t* stg = sm;                                               // [kS][A stage | B panel step]
  float* hx = reinterpret_cast<float*>(stg + (size_t)kS * M::kStage);  // gate/up: [4][kMaxTok][32]
  uint64_t* bars = reinterpret_cast<uint64_t*>(reinterpret_cast<uint8_t*>(hx) + M::kEpiSmem);
  uint64_t* full = bars;                  // both operands of the stage landed (two producers)
  uint64_t* empty = full + kS;            // the MMAs reading the stage completed
  uint64_t* ready = empty + kS;           // the stage's scale factors are in TMEM set s (4 warps x 32)
  uint64_t* accfull = ready + kS;         // [kBufs] every MMA lane's part of the buffer's unit completed
  uint64_t* accempty = accfull + 2;       // [kBufs]
  uint32_t* tslot = reinterpret_cast<uint32_t*>(accempty + 2);  // [0] TMEM address, [1] abort flag
  volatile int* abort = reinterpret_cast<volatile int*>(tslot + 1);
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
  // the tensor copies write the first 8 bytes of every 16-byte operand row;
  // the other 8 stay as set here
  for (int c = tid; c < kS * 2 * (kAOp / 16); c += kThr)
    *reinterpret_cast<uint2*>(stg + (size_t)(c / (2 * (kAOp / 16))) * M::kStage +
                              (size_t)((c / (kAOp / 16)) & 1) * kAOp + 16 * (c % (kAOp / 16)) + 8) =
        make_uint2(0u, 0u);
  tc::fence_proxy_async();
  if (tid == 0) {
    *abort = 0;
    for (int s = 0; s < kS; ++s) {
      mbar_init(&full[s], 2);
      mbar_init(&empty[s], kMma);
      mbar_init(&ready[s], 128);
    }
    for (int a = 0; a < kBufs; ++a) {
      mbar_init(&accfull[a], kMma);
      mbar_init(&accempty[a], kEpiThreads);
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
      Cursor<kDown> ca, cp;
      ca.i = cp.i = 0;
      ca.ks = cp.ks = 0;
      ca.g = cp.g = tc_unit<kDown>(p, st, b0);
      // weight blocks are read once: start them towards L2 kPf steps before their tensor copy
      auto prefetch = [&]() {
        prefetch_l2(cp.g.w + (size_t)cp.ks * kTcPairBytes, kTcPairBytes);
        cursor_next<kDown>(p, st, cp, n_units);
      };
      for (int q = 0; q < M::kPf && cp.i < n_units; ++q) prefetch();
      for (int j = 0; ca.i < n_units; ++j) {
        const int s = j % kS;
        if (j >= kS && !tc::bounded_wait_sleep(&empty[s], (uint32_t)((j / kS - 1) & 1), p.status, abort)) break;
        uint8_t* sb = stg + (size_t)s * M::kStage;
        // both tiles' 2 x 8,192 code bytes (counted as read from global memory) + 1,024 scale bytes
        mbar_arrive_expect_tx(&full[s], (uint32_t)kTcPairBytes);
        tc::tma_load_2d(sb, &wmap, 0, ca.g.y + ca.ks * kCmRows, &full[s]);
        bulk_g2s(sb + 2 * kAOp, ca.g.w + (size_t)ca.ks * kTcPairBytes + 2 * kTcCodeBytes, 1024, &full[s]);
        if (M::kPf > 0 && cp.i < n_units) prefetch();
        cursor_next<kDown>(p, st, ca, n_units);
      }
    }
  } else if (warp == kPanelWarp) {
    if (lane == 0) {
      Cursor<kDown> cb;
      cb.i = 0;
      cb.ks = 0;
      cb.g = tc_unit<kDown>(p, st, b0);
      // panels of every slot use the stride of the largest K step count
      const int pstride = kDown ? tc_ksteps(p.F > p.S ? p.F : p.S) : tc_ksteps(p.d);
      for (int j = 0; cb.i < n_units; ++j) {
        const int s = j % kS;
        if (j >= kS && !tc::bounded_wait_sleep(&empty[s], (uint32_t)((j / kS - 1) & 1), p.status, abort)) break;
        const int N = M::kPlanes * npad_of(cb.g.n);
        uint8_t* sb = stg + (size_t)s * M::kStage + M::kAPair;
        const uint8_t* src = (kDown ? p.hpanel : p.xpanel) + ((size_t)cb.g.panel * pstride + cb.ks) * M::kPanelStep;
        // N rows and their scale words right behind them
        mbar_arrive_expect_tx(&full[s], (uint32_t)(N * kTcStepK + 512 * M::kSfBlocks));
        bulk_g2s(sb, src, (uint32_t)(N * kTcStepK + 512 * M::kSfBlocks), &full[s]);
        cursor_next<kDown>(p, st, cb, n_units);
      }
    }
  } else if (warp >= kMmaWarp0 && warp < kMmaWarp0 + kMma) {
    if (lane == 0) {
      const int t = warp - kMmaWarp0;  // M tile t of every unit
      int j0 = 0;                      // first K step of unit i
      bool ok = true;
      for (int i = 0; i < n_units && ok; ++i) {
        const TcUnit g = tc_unit<kDown>(p, st, b0 + i * G);
        const int N = M::kPlanes * npad_of(g.n), acc = i % kBufs;
        const bool mine = t < g.nt;  // a pair of one tile leaves lane 1 without MMAs
        if (i >= kBufs && !tc::bounded_wait(&accempty[acc], (uint32_t)((i / kBufs - 1) & 1), p.status, abort)) break;
        tc::fence_after();
        const uint32_t d = tmem + M::kDCol * (kMma * acc + t);
        for (int ks = 0; ks < g.nks; ++ks) {
          const int jj = j0 + ks, s = jj % kS;
          // every lane takes part in every step's hand-off, with or without MMAs
          if (!tc::bounded_wait(&ready[s], (uint32_t)((jj / kS) & 1), p.status, abort)) {  // operands landed, scales in TMEM
            ok = false;
            break;
          }
          tc::fence_after();
          if (mine) {
            const uint8_t* ab = stg + (size_t)s * M::kStage + (size_t)t * kAOp;
            const uint8_t* bb = stg + (size_t)s * M::kStage + M::kAPair;
            const uint32_t sf = tmem + kSfCol + kSfSet * s;
#pragma unroll
            for (int kb = 0; kb < 4; ++kb) {
              const uint64_t ad = tc::smem_desc(ab + 2 * kb * 128, 128, 8 * 128);
              const uint64_t bd = tc::smem_desc(bb + 2 * kb * 128, 128, 8 * 128);
              tc::mma_mxf4_mxf8(d, ad, bd, tc::idesc_mxf4_mxf8(128, N, kb, kb), sf + 8 * t, sf + 16,
                                (ks > 0 || kb > 0) ? 1u : 0u);
            }
          }
          tc::commit(&empty[s]);
        }
        if (!ok) break;
        tc::commit(&accfull[acc]);
        j0 += g.nks;
      }
    }
  } else if (warp >= kSfWarp0 && warp < kSfWarp0 + 4) {
    // scale factors of every stage into TMEM set s, in the warp's lane
    // quadrant (each quadrant holds the same copy): SFA words [lane][4] of M
    // tile 0 / 1 to columns +0 / +8, SFB to +16 (+4 per 512-byte block)
    const uint32_t qbase = tmem + ((uint32_t)((warp & 3) * 32) << 16) + kSfCol;
    int j = 0;
    bool ok = true;
    for (int i = 0; i < n_units && ok; ++i) {
      const TcUnit g = tc_unit<kDown>(p, st, b0 + i * G);
      for (int ks = 0; ks < g.nks; ++ks, ++j) {
        const int s = j % kS;
        // the warp's lanes leave together (one lane's verdict), so tcgen05.st stays warp-uniform
        ok = __shfl_sync(0xffffffffu, tc::bounded_wait(&full[s], (uint32_t)((j / kS) & 1), p.status, abort) ? 1 : 0, 0) != 0;
        if (!ok) break;
        const uint8_t* sb = stg + (size_t)s * M::kStage;
        const uint8_t* sbf = sb + M::kAPair + M::kPlanes * npad_of(g.n) * kTcStepK;  // SFB behind the N rows
        const uint4 wa0 = *reinterpret_cast<const uint4*>(sb + 2 * kAOp + 16 * lane);
        const uint4 wb0 = *reinterpret_cast<const uint4*>(sbf + 16 * lane);
        tc::fence_after();
        const uint32_t sf = qbase + kSfSet * s;
        tc::st4(sf, wa0.x, wa0.y, wa0.z, wa0.w);
        if (g.nt > 1) {
          const uint4 wa1 = *reinterpret_cast<const uint4*>(sb + 2 * kAOp + 512 + 16 * lane);
          tc::st4(sf + 8, wa1.x, wa1.y, wa1.z, wa1.w);
        }
        tc::st4(sf + 16, wb0.x, wb0.y, wb0.z, wb0.w);
        if (M::kSfBlocks > 1) {
          const uint4 wb1 = *reinterpret_cast<const uint4*>(sbf + 512 + 16 * lane);
          tc::st4(sf + 20, wb1.x, wb1.y, wb1.z, wb1.w);
        }
        tc::wait_st();
        tc::fence_before();
        mbar_arrive(&ready[s]);
      }
    }
  } else if (warp >= kEpiWarp0) {
    // epilogue: warp w reads TMEM lanes 32 (w % 4) .. +31; the warps of a
    // quadrant take 16-column chunks in turn
    const int qd = warp & 3, eg = (warp - kEpiWarp0) >> 2, ew = warp - kEpiWarp0, et = tid - kEpiWarp0 * 32;
    const uint32_t trow = tmem + ((uint32_t)(qd * 32) << 16);
    // gate/up: TMEM lane l of a quadrant is f offset kk(l) within its 32-element block
    const int kk = 8 * ((lane & 15) >> 2) + 4 * (lane >> 4) + (lane & 3);
    const int pstride = tc_ksteps(p.F > p.S ? p.F : p.S);
    for (int i = 0; i < n_units; ++i) {
      const TcUnit g = tc_unit<kDown>(p, st, b0 + i * G);
      const int npad = npad_of(g.n), acc = i % kBufs;
      // every epilogue thread leaves on the same verdict: the named barriers below need all 256
      const bool ok = tc::bounded_wait_sleep(&accfull[acc], (uint32_t)((i / kBufs) & 1), p.status, abort);
      // one verdict for all 256 (the abort flag may rise between two threads' reads of it)
      if (named_bar_or(1, kEpiThreads, !ok || *abort)) break;
      tc::fence_after();
      if (kDown) {  // part rows q0 + m, column 128 (mt + t) + 32 qd + lane: the sum of the 4 planes
        for (int t = 0; t < g.nt; ++t) {
          const int row = 128 * (g.mt + t) + 32 * qd + lane;
          const uint32_t dcol = trow + M::kDCol * (kMma * acc + t);
          for (int c0 = 16 * eg; c0 < npad; c0 += 16 * kEpiPerQuad) {
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
        }
        tc::fence_before();
        mbar_arrive(&accempty[acc]);
      } else {
        for (int t = 0; t < g.nt; ++t) {
          const int mt = g.mt + t;
          // 1. accumulator of M tile mt -> hx[block][token][f offset]: blocks 0, 1 gate, 2, 3 up
          named_bar(1, kEpiThreads);  // the previous readers of hx are done
          const uint32_t dcol = trow + M::kDCol * (kMma * acc + t);
          for (int c0 = 16 * eg; c0 < npad; c0 += 16 * kEpiPerQuad) {
            float v[16], w[16];
            tc::ld16(dcol + c0, v);
            tc::ld16(dcol + npad + c0, w);
#pragma unroll
            for (int x = 0; x < 16; ++x)
              if (c0 + x < npad) hx[(qd * kMaxTok + c0 + x) * 32 + kk] = v[x] + w[x];
          }
          if (t == g.nt - 1) {
            tc::fence_before();
            mbar_arrive(&accempty[acc]);  // every accumulator of the unit has been read
          }
          named_bar(1, kEpiThreads);
          // 2. h = SiLU(gate) * up, four MXFP8 planes, straight into the down step's
          // h panel: f block 2 mt + b is K step mt / 2, elements 64 (mt % 2) + 32 b ..
          uint8_t* dst = p.hpanel + ((size_t)g.panel * pstride + (mt >> 1)) * kTcPanelStepD;
          const int kh = 64 * (mt & 1), nblk = g.f / 32;
          for (int it = ew; it < 2 * npad; it += kEpiThreads / 32) {
            const int m = it >> 1, b = it & 1;
            float h = 0.f;
            if (m < g.n && 2 * mt + b < nblk) {
              const float gate = hx[(b * kMaxTok + m) * 32 + lane], up = hx[((2 + b) * kMaxTok + m) * 32 + lane];
              h = gate / (1.f + __expf(-gate)) * up;
            }
            uint32_t code[4], sc[4];
            tc::split_planes4_fixed(h, code, sc);
            const int k = kh + 32 * b + lane;
#pragma unroll
            for (int pl = 0; pl < 4; ++pl) {
              const int row = pl * npad + m;
              dst[((row >> 3) * 8 + (k >> 4)) * 128 + (row & 7) * 16 + (k & 15)] = (uint8_t)code[pl];
            }
            if (lane < 4) {
              const uint32_t sv = lane == 0 ? sc[0] : lane == 1 ? sc[1] : lane == 2 ? sc[2] : sc[3];
              dst[hsf_off(npad, lane * npad + m, 2 * (mt & 1) + b)] = (uint8_t)sv;
            }
          }
          // 3. scale bytes of the rows past the 4 planes (127), and the half K step
          // past the last M tile when the tile count is odd (codes 0, scales 127)
          for (int o = et; o < 2 * (256 - 4 * npad); o += kEpiThreads)
            dst[hsf_off(npad, 4 * npad + (o >> 1), 2 * (mt & 1) + (o & 1))] = 127;
          if ((mt & 1) == 0 && mt + 1 == tc_msteps(g.f)) {
            for (int o = et; o < 4 * npad * 4; o += kEpiThreads) {
              const int row = o >> 2, kc = 4 + (o & 3);
              *reinterpret_cast<uint4*>(dst + ((row >> 3) * 8 + kc) * 128 + (row & 7) * 16) = make_uint4(0, 0, 0, 0);
            }
            for (int o = et; o < 2 * 256; o += kEpiThreads) dst[hsf_off(npad, o >> 1, 2 + (o & 1))] = 127;
          }
        }
      }
    }
  }
  tc::fence_before();
  __syncthreads();
  if (warp == 0) {
    if (*abort) {  // the roles stopped early: let every copy and MMA already issued finish
      const uint64_t t0 = globaltimer();
      while ((long long)(globaltimer() - t0) < tc::kDrainNs) __nanosleep(10000);
    }
    tc::fence_after();
    tc::dealloc(tmem, kTmemCols);
  }
}

// Activation panels: one CTA per (panel, kPanelSteps K steps). Panel rows
// n < 2 npad: plane n / npad, token m = n % npad of the block (rows past the
// block's tokens are zero, their scales 127). The rows' tokens are looked up
// once into shared memory; then every thread issues all of its 16-byte loads
// of the block's K steps before its first store, so the block waits for one
// round trip, not one per chunk.
constexpr int kPanelSteps = 4;  // K steps of the x panels per block
constexpr int kPanelThreads = 256;
constexpr int kPanelLoads = (2 * kMaxTok * 8 * kPanelSteps + kPanelThreads - 1) / kPanelThreads;  // per thread
__global__ void __launch_bounds__(kPanelThreads) pack_panels_kernel(FwdParams p) {
  pdl_enter();
  __shared__ int tok[2 * kMaxTok];  // token of each panel row, -1 for padding rows
  const int pb = blockIdx.x;
  const int ns = *p.n_slots;
  if (pb >= p.panel_prefix[ns]) return;
  const int s = find_unit_slot(p.panel_prefix, ns, pb);
  const int tb = pb - p.panel_prefix[s];
  const int n = min(kMaxTok, p.slot_n[s] - kMaxTok * tb), q0 = p.slot_q0[s] + kMaxTok * tb, npad = npad_of(n);
  const int nks = tc_ksteps(p.d);
  for (int r = threadIdx.x; r < 2 * npad; r += kPanelThreads) {
    const int m = r - (r >= npad ? npad : 0);
    tok[r] = m < n ? tok_of(p, q0 + m) : -1;
  }
  __syncthreads();
  const int ks0 = blockIdx.y * kPanelSteps, nk = min(nks, ks0 + kPanelSteps) - ks0;
  const int nch = 2 * npad * 8;  // 16-byte chunks (row, kc) of one K step's N = 2 npad rows
  uint4 v[kPanelLoads];
#pragma unroll
  for (int i = 0; i < kPanelLoads; ++i) {
    const int o = threadIdx.x + kPanelThreads * i, kk = o / nch, c = o - kk * nch;
    const int row = c >> 3, k0 = kTcStepK * (ks0 + kk) + 16 * (c & 7);
    const int t = kk < nk ? tok[row] : -1;
    v[i] = make_uint4(0, 0, 0, 0);
    if (t >= 0 && k0 < p.d64)
      v[i] = __ldg(reinterpret_cast<const uint4*>(p.xq + ((size_t)t * 2 + (row >= npad)) * p.d64 + k0));
  }
#pragma unroll
  for (int i = 0; i < kPanelLoads; ++i) {
    const int o = threadIdx.x + kPanelThreads * i, kk = o / nch, c = o - kk * nch;
    if (kk >= nk) continue;
    const int row = c >> 3, kc = c & 7;
    uint8_t* dst = p.xpanel + ((size_t)pb * nks + ks0 + kk) * kTcPanelStep;
    *reinterpret_cast<uint4*>(dst + ((row >> 3) * 8 + kc) * 128 + (row & 7) * 16) = v[i];
  }
  if (threadIdx.x < 128) {  // scale word (lane l, r) for B row 32 r + l, every K step of the block
    const int l = threadIdx.x >> 2, r = threadIdx.x & 3, row = 32 * r + l;
    const int t = row < 2 * npad ? tok[row] : -1;
    const uint8_t* sc = t >= 0 ? p.xqs + ((size_t)t * 2 + (row >= npad)) * p.xq_spitch : nullptr;
    for (int kk = 0; kk < nk; ++kk) {
      const int ks = ks0 + kk;
      uint32_t w = 0x7F7F7F7Fu;
      if (sc) {
        w = 0;
        for (int kb = 0; kb < 4; ++kb) {
          const int blk = 4 * ks + kb;
          w |= (uint32_t)(blk < p.xq_spitch ? sc[blk] : 127) << (8 * kb);
        }
      }
      *reinterpret_cast<uint32_t*>(p.xpanel + ((size_t)pb * nks + ks) * kTcPanelStep + 2 * npad * kTcStepK + 16 * l + 4 * r) = w;
    }
  }
}

// The tcgen05 weight copies: one thread per (expert, M tile, K step, M row).
// Gate/up: M row m of tile a is row m % 16 of pair tile 4a + (m / 16) % 4
// (gate rows for m < 64, up rows after), K = d. Down: row 128a + m of the
// down matrix, K = f.
__global__ void repack_tc_kernel(const uint8_t* codes, const uint8_t* scales, int n_exp, int d, int f,
                                 size_t ccs, size_t css, uint8_t* out, size_t out_stride, bool down, int* err) {
  // every tile of the pairs, the second tile of an odd last pair included (all code 0, scale 127)
  const int nms = 2 * (down ? tc_dn_pairs(d) : tc_gu_pairs(f)), K = down ? f : d, nks = tc_ksteps(K);
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
    uint8_t* dst = out + (size_t)x * out_stride + ((size_t)(a >> 1) * nks + ks) * kTcPairBytes;
    uint8_t* dcode = dst + (size_t)(a & 1) * kTcCodeBytes;
    for (int kc = 0; kc < 8; ++kc) {
      const int k0 = kTcStepK * ks + 16 * kc;
      uint2 v = make_uint2(0u, 0u);
      if (live && k0 < K) {
        uint8_t b[8];
        for (int i = 0; i < 8; ++i) b[i] = cr[k0 / 2 + i];
        v.x = (uint32_t)b[0] | ((uint32_t)b[1] << 8) | ((uint32_t)b[2] << 16) | ((uint32_t)b[3] << 24);
        v.y = (uint32_t)b[4] | ((uint32_t)b[5] << 8) | ((uint32_t)b[6] << 16) | ((uint32_t)b[7] << 24);
      }
      *reinterpret_cast<uint2*>(dcode + ((m >> 3) * 8 + kc) * 64 + (m & 7) * 8) = v;
    }
    uint32_t w = 0;
    for (int kb = 0; kb < 4; ++kb) {
      const int blk32 = 4 * ks + kb;
      const uint32_t sc = (live && 32 * blk32 < K) ? sr[blk32] : 127u;
      if (sc == 255u) atomicExch(err, 1);
      w |= sc << (8 * kb);
    }
    *reinterpret_cast<uint32_t*>(dst + 2 * kTcCodeBytes + 512 * (a & 1) + 16 * (m & 31) + 4 * (m >> 5)) = w;
  }
}

// x as two E4M3 planes per 32-element block (what split_planes<2> computes
// for one element per lane), four threads per block of 32: each thread loads
// 8 bf16 at once, the block maximum of each plane comes from two shuffles
// within the four, and every thread stores its 8 codes per plane in one 8-byte
// store. The bits equal the one-element-per-lane form (the same maxima and
// conversions).
__global__ void __launch_bounds__(256) prep_xq_kernel(FwdParams p) {
  pdl_enter();
  const int g = blockIdx.x * blockDim.x + threadIdx.x, sub = g & 3;
  const int nb = p.xq_spitch;  // blocks per row, scale padding included
  if (g >= p.T * nb * 4) return;  // whole groups of four: T nb 4 and the block size are multiples of 4
  const int item = g >> 2, t = item / nb, b = item - t * nb;
  uint8_t* qs = p.xqs + (size_t)t * 2 * p.xq_spitch + b;
  if (32 * b >= p.d64) {  // scale padding
    if (sub == 0) {
      qs[0] = 127;
      qs[p.xq_spitch] = 127;
    }
    return;
  }
  const int k0 = 32 * b + 8 * sub;
  // the four threads of a block take every branch together (the exits above are per block): the
  // shuffles name just them
  const unsigned gmask = 0xFu << (threadIdx.x & 28);
  float v[8];
  if (k0 < p.d) {
    const uint4 xv = *reinterpret_cast<const uint4*>(p.x + (size_t)t * p.d + k0);
    const uint32_t w4[4] = {xv.x, xv.y, xv.z, xv.w};
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      v[2 * q] = __uint_as_float(w4[q] << 16);
      v[2 * q + 1] = __uint_as_float(w4[q] & 0xFFFF0000u);
    }
  } else {
#pragma unroll
    for (int q = 0; q < 8; ++q) v[q] = 0.f;
  }
  uint8_t* qh = p.xq + (size_t)t * 2 * p.d64 + k0;
#pragma unroll
  for (int pl = 0; pl < 2; ++pl) {
    float amax = 0.f;
#pragma unroll
    for (int q = 0; q < 8; ++q) amax = fmaxf(amax, fabsf(v[q]));
    amax = fmaxf(amax, __shfl_xor_sync(gmask, amax, 1));
    amax = fmaxf(amax, __shfl_xor_sync(gmask, amax, 2));
    int sh = amax > 0.f ? (int)((__float_as_uint(amax) >> 23) & 0xFF) - 127 - 7 : 0;
    sh = max(-127, min(127, sh));
    const float ish = __uint_as_float((uint32_t)(127 - sh) << 23), fsh = __uint_as_float((uint32_t)(127 + sh) << 23);
    uint32_t codes[2] = {0u, 0u};
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      uint16_t c2;  // low byte: element 2q, high byte: element 2q + 1
      asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(c2) : "f"(v[2 * q + 1] * ish), "f"(v[2 * q] * ish));
      uint32_t h2;
      asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(h2) : "h"(c2));
      v[2 * q] -= __half2float(__ushort_as_half((unsigned short)(h2 & 0xFFFFu))) * fsh;
      v[2 * q + 1] -= __half2float(__ushort_as_half((unsigned short)(h2 >> 16))) * fsh;
      codes[q >> 1] |= (uint32_t)c2 << (16 * (q & 1));
    }
    *reinterpret_cast<uint2*>(qh + (size_t)pl * p.d64) = make_uint2(codes[0], codes[1]);
    if (sub == 0) qs[(size_t)pl * p.xq_spitch] = (uint8_t)(sh + 127);
  }
}

}  // namespace

cudaError_t launch_repack_tc(const uint8_t* codes, const uint8_t* scales, int n_exp, int d, int f,
                             size_t canon_code_stride, size_t canon_scale_stride, uint8_t* out, size_t out_stride,
                             bool down, int* err_flag, cudaStream_t stream) {
  repack_tc_kernel<<<1024, 256, 0, stream>>>(codes, scales, n_exp, d, f, canon_code_stride, canon_scale_stride, out,
                                             out_stride, down, err_flag);
  return cudaGetLastError();
}

cudaError_t configure_tcgemm(int max_smem) {
  cudaError_t e = cudaFuncSetAttribute(gemm_tc_kernel<false>, cudaFuncAttributeMaxDynamicSharedMemorySize, max_smem);
  if (e == cudaSuccess)
    e = cudaFuncSetAttribute(gemm_tc_kernel<true>, cudaFuncAttributeMaxDynamicSharedMemorySize, max_smem);
  return e;
}

cudaError_t launch_panels_tc(const FwdParams& p, cudaStream_t stream) {
  launch_chained(prep_xq_kernel, dim3((p.T * p.xq_spitch * 4 + 255) / 256), dim3(256), 0, stream, p);
  // panels: at most ceil(Q / 48) + slots blocks (the kernels skip the ones past the count)
  const int max_panels = (p.P + p.T) / kTcGemmRows + p.E + 2;
  return launch_chained(pack_panels_kernel, dim3(max_panels, (tc_ksteps(p.d) + kPanelSteps - 1) / kPanelSteps),
                        dim3(256), 0, stream, p);
}

cudaError_t launch_gemm_gateup_tc(const FwdParams& p, cudaStream_t stream, int num_sms) {
  const size_t smem = tc_gemm_smem_bytes(p.E, false);
  return launch_chained(gemm_tc_kernel<false>, dim3(num_sms), dim3(kThr), smem, stream, p,
                        *static_cast<const CUtensorMap*>(p.tmap_gu));
}

cudaError_t launch_gemm_down_tc(const FwdParams& p, cudaStream_t stream, int num_sms) {
  const size_t smem = tc_gemm_smem_bytes(p.E, true);
  return launch_chained(gemm_tc_kernel<true>, dim3(num_sms), dim3(kThr), smem, stream, p,
                        *static_cast<const CUtensorMap*>(p.tmap_dn));
}

size_t tc_gemm_smem_bytes(int E, bool down) {
  return (down ? tc_smem_fixed<true>() : tc_smem_fixed<false>()) + tc_table_bytes(E);
}

// The weight copy as a 2-D tensor of "16 x U4, 16-byte aligned" elements:
// rows of 128 codes (64 bytes: one core matrix of 8 rows x 16 codes), so that
// a box of 256 rows is the 2 x 8,192 code bytes of a tile pair's block and a
// box of 128 rows one tile's, widened on the way into shared memory.
// The same copy as a 3-D tensor (rows of 64 bytes, groups of 16 rows) with a
// box of 128 x 16 x 17: the whole 17,408-byte block of a tile pair's K step --
// both tiles' codes and their 1,024 scale bytes -- in one tensor copy, every
// 8 bytes widened to 16 (the scale bytes too, which their readers skip over).
bool encode_tc_block_map(const void* base, size_t bytes, void* map) {
  static PFN_cuTensorMapEncodeTiled_v12000 encode = nullptr;
  if (!encode) {
    void* fn = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q) != cudaSuccess ||
        q != cudaDriverEntryPointSuccess || !fn)
      return false;
    encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
  }
  if (bytes % kTcPairBytes != 0 || bytes / 1024 >= (1ull << 31)) return false;
  const cuuint64_t dims[3] = {128, 16, (cuuint64_t)(bytes / 1024)}, strides[2] = {64, 1024};
  const cuuint32_t box[3] = {128, 16, kTcPairBytes / 1024}, es[3] = {1, 1, 1};
  return encode(static_cast<CUtensorMap*>(map), CU_TENSOR_MAP_DATA_TYPE_16U4_ALIGN16B, 3, const_cast<void*>(base), dims,
                strides, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
                CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

bool encode_tc_weight_map(const void* base, size_t bytes, void* map, int box_rows) {
  static PFN_cuTensorMapEncodeTiled_v12000 encode = nullptr;
  if (!encode) {
    void* fn = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q) != cudaSuccess ||
        q != cudaDriverEntryPointSuccess || !fn)
      return false;
    encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
  }
  if (bytes % 64 != 0 || bytes / 64 >= (1ull << 31)) return false;
  const cuuint64_t dims[2] = {128, (cuuint64_t)(bytes / 64)}, strides[1] = {64};
  if (box_rows != 128 && box_rows != 256) return false;
  const cuuint32_t box[2] = {128, (cuuint32_t)box_rows}, es[2] = {1, 1};
  return encode(static_cast<CUtensorMap*>(map), CU_TENSOR_MAP_DATA_TYPE_16U4_ALIGN16B, 2, const_cast<void*>(base), dims,
                strides, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
                CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace moe
