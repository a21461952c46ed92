// Gate/up + SwiGLU of the general path on the 5th-generation tensor cores:
// a block-scaled MMA of the MXFP4 expert weights (E2M1 codes with their E8M0
// scales, exactly as stored) by MXFP8 activations (tcgen05.mma
// kind::mxf8f6f4.block_scale), accumulators in tensor memory.
//
// The activation x (bf16) enters as two MXFP8 planes, x = 2^sh * hi + 2^sl * lo
// per 32-element block (E4M3 codes hi and lo with their own E8M0 scales): a
// bf16 value has 8 significant bits, hi keeps its top 4 and lo the remaining 4,
// so the split is exact except for elements below about 2^-10 of their block's
// largest one. Token t of a unit is B row t (hi) and B row npad + t (lo); its
// gate (up) value is D[., t] + D[., npad + t].
//
// Work unit: (slot, 4 consecutive 16-row pair tiles = 64 f-values, block of
// up to 48 tokens of the slot). The M = 128 tile holds the 64 gate rows, then
// the 64 up rows, in pair-tile row order; N = 2 * npad (npad = tokens rounded
// up to 8, at least 8); K = d in steps of 128 (two 64-element k tiles, four
// K=32 MMAs). A CTA (4 warps) loops over units; every thread copies its share
// of each stage (weight codes in 4-byte pieces from the packed tiles into the
// padded MXFP4 operand layout, x planes in 16-byte pieces, raw scale bytes)
// with cp.async, three stages in flight; the warps then write the stage's
// scale factors to tensor memory, and one thread issues the stage's MMAs and
// commits them to the stage's mbarrier, which frees the buffers. After a
// unit's last stage the four warps read the accumulators (warp w: rows
// 32w..32w+31), the up warps hand their values to the gate warps through
// shared memory, and the gate warps write h = SiLU(gate) * up in the f16
// hi + lo format of the down step.
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

constexpr int kThr = 512;                 // 16 warps; warp w reaches TMEM lane quadrant w % 4
constexpr int kStages = 7;                // stages of raw weights + x planes in flight
constexpr int kStageK = 128;              // K elements per stage: two 64-element k tiles
constexpr int kMaxTok = kTcGemmRows;      // tokens per unit
constexpr int kMaxN = 2 * kMaxTok;        // B rows: hi and lo planes
constexpr int kRaw = 16 * kTileBytes;     // 8 packed tiles x 2 k tiles, as stored (codes + scales)
constexpr int kBStage = kMaxN * kStageK;  // E4M3, already in the operand layout
constexpr int kSfbRaw = kMaxN * 4;        // 4 K blocks per B row
constexpr int kStageBytes = kRaw + kBStage + kSfbRaw;
constexpr int kAStage = 128 * kStageK;    // padded MXFP4 operand: 16 bytes per 16 elements (2 buffers)
constexpr uint32_t kTmemCols = 256;       // D: columns [0, 96); scale-factor sets from column 128
constexpr int kSfCol = 128;               // set s (step parity): SFA columns 128 + 16s .. +3, SFB +8 .. +10
constexpr long long kWaitNs = 50000000LL;

__device__ __forceinline__ void cpa4(void* dst, const void* src) {
  asm volatile("cp.async.ca.shared.global [%0], [%1], 4;" ::"r"(smem_u32(dst)), "l"(src) : "memory");
}
__device__ __forceinline__ void cpa16(void* dst, const void* src) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(smem_u32(dst)), "l"(src) : "memory");
}
__device__ __forceinline__ void cp_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_wait() {
  asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
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

struct TcUnit {
  int e, f;     // expert (E = shared) and its ffn
  int q0, n;    // first h row and tokens of the block
  int tau0;     // first pair tile
};

__device__ __forceinline__ TcUnit tc_unit(const FwdParams& p, int u) {
  const int ns = *p.n_slots;
  const int s = find_unit_slot(p.gu_prefix, ns, u);
  const int r = u - p.gu_prefix[s];
  TcUnit g;
  g.e = p.slot_expert[s];
  g.f = (g.e == p.E) ? p.S : p.F;
  const int ngrp = (g.f / 16 + 3) / 4;
  const int tb = r / ngrp, grp = r - tb * ngrp;
  g.q0 = p.slot_q0[s] + kMaxTok * tb;
  g.n = min(kMaxTok, p.slot_n[s] - kMaxTok * tb);
  g.tau0 = 4 * grp;
  return g;
}

__device__ __forceinline__ int tok_of(const FwdParams& p, int q) { return q < p.P ? p.perm[q] / p.k : q - p.P; }

// The copies of one stage, in a fixed thread mapping so that every address is
// a per-unit base plus a per-thread constant:
//  * weights: the 16 (tile, k tile) areas of 544 bytes, as stored, in
//    16-byte pieces (piece o = tid + 128 i);
//  * x planes: thread tid copies 16-code chunk tid & 7 of B rows
//    (tid >> 3) + (kThr / 8) j straight into the operand layout, and the 4
//    scale bytes of B row tid.
constexpr int kBRowsPerThread = (kMaxN * 8 + kThr - 1) / kThr;

struct Loader {
  int unit_i, ks, nks, n_units, K64;
  const uint8_t* wbase;  // packed tile (pair tile tau0, k tile 0)
  int ntile_valid;       // pair tiles of the unit that exist (1..4)
  int n2;                // B rows 2n
  const uint8_t* xrow[kBRowsPerThread];  // this thread's B rows (chunk tid & 7 folded in)
  int xdst[kBRowsPerThread];
  const uint8_t* srow;   // scale row of B row tid (or null)
  int sdst;
};

__device__ void loader_unit(const FwdParams& p, Loader& ld) {
  const TcUnit g = tc_unit(p, blockIdx.x + ld.unit_i * gridDim.x);
  ld.wbase = p.packed + (size_t)g.e * p.expert_stride + (size_t)g.tau0 * ld.K64 * 2 * kTileBytes;
  ld.ntile_valid = min(4, g.f / 16 - g.tau0);
  ld.n2 = 2 * g.n;
  const int npad = max(8, (g.n + 7) & ~7);
  const int kc = threadIdx.x & 7;
#pragma unroll
  for (int j = 0; j < kBRowsPerThread; ++j) {
    const int rowp = (threadIdx.x >> 3) + (kThr / 8) * j;
    if (rowp < ld.n2) {
      const int plane = rowp >= g.n, m = rowp - plane * g.n, n = plane * npad + m;
      ld.xrow[j] = p.xq + ((size_t)tok_of(p, g.q0 + m) * 2 + plane) * p.d64 + 16 * kc;
      ld.xdst[j] = kRaw + ((n >> 3) * 8 + kc) * 128 + (n & 7) * 16;
    } else {
      ld.xrow[j] = nullptr;
    }
  }
  const int rowp = threadIdx.x;
  if (rowp < ld.n2) {
    const int plane = rowp >= g.n, m = rowp - plane * g.n, n = plane * npad + m;
    ld.srow = p.xqs + ((size_t)tok_of(p, g.q0 + m) * 2 + plane) * p.xq_spitch;
    ld.sdst = kRaw + kBStage + 4 * n;
  } else {
    ld.srow = nullptr;
  }
}

__device__ void loader_init(const FwdParams& p, Loader& ld, int n_units) {
  ld.unit_i = 0;
  ld.ks = 0;
  ld.n_units = n_units;
  ld.K64 = k64_tiles(p.d);
  ld.nks = (ld.K64 + 1) / 2;
  loader_unit(p, ld);
}

// Copy the loader's next stage into buffer `sb` and advance.
__device__ void loader_issue(const FwdParams& p, Loader& ld, uint8_t* sb) {
  if (ld.unit_i >= ld.n_units) return;
  const int K64 = ld.K64, ks = ld.ks;
  const int nkt = min(2, K64 - 2 * ks);
  const size_t rowstride = (size_t)K64 * 2 * kTileBytes;  // one pair tile
  const uint8_t* w0 = ld.wbase + (size_t)ks * 2 * 2 * kTileBytes;
  constexpr int kPieces = kTileBytes / 16;  // 34 per area
#pragma unroll
  for (int i = 0; i < (16 * kPieces + kThr - 1) / kThr; ++i) {
    const int o = threadIdx.x + kThr * i;
    if (o >= 16 * kPieces) break;
    const int tk = o / kPieces, pc = o - tk * kPieces, t = tk >> 1, kts = tk & 1;
    if ((t & 3) >= ld.ntile_valid || kts >= nkt) continue;
    cpa16(sb + tk * kTileBytes + 16 * pc,
          w0 + (t & 3) * rowstride + (t >> 2) * kTileBytes + kts * 2 * kTileBytes + 16 * pc);
  }
  const bool full_stage = nkt == 2 || (threadIdx.x & 7) < 4;  // a single-k-tile stage has 4 chunks per row
#pragma unroll
  for (int j = 0; j < kBRowsPerThread; ++j)
    if (ld.xrow[j] && full_stage) cpa16(sb + ld.xdst[j], ld.xrow[j] + (size_t)ks * kStageK);
  if (ld.srow) cpa4(sb + ld.sdst, ld.srow + 4 * ks);
  if (++ld.ks == ld.nks) {
    ld.ks = 0;
    if (++ld.unit_i < ld.n_units) loader_unit(p, ld);
  }
}

__global__ void __launch_bounds__(kThr, 1) gemm_gateup_tc_kernel(FwdParams p) {
  extern __shared__ __align__(1024) uint8_t sm[];
  uint8_t* stages = sm;
  uint8_t* abuf = sm + (size_t)kStages * kStageBytes;                  // 2 padded MXFP4 operand buffers
  uint8_t* bbuf = abuf + 2 * kAStage;                                   // 2 MXFP8 operand buffers
  float* upx = reinterpret_cast<float*>(bbuf + 2 * kBStage);           // [64 rows][kMaxTok]
  uint64_t* bars = reinterpret_cast<uint64_t*>(upx + 64 * kMaxTok);   // empty[kStages], done
  uint32_t* tslot = reinterpret_cast<uint32_t*>(bars + kStages + 1);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int total = p.gu_prefix[*p.n_slots];
  const int n_units = total > (int)blockIdx.x ? (total - (int)blockIdx.x + gridDim.x - 1) / gridDim.x : 0;
  if (n_units == 0) return;
  // zero the stage buffers once: the padding half of every MXFP4 operand row
  // stays zero, and rows a unit does not fill hold finite values
  for (int o = tid; o < (kStages * kStageBytes + 2 * kAStage + 2 * kBStage) / 16; o += kThr)
    reinterpret_cast<uint4*>(stages)[o] = make_uint4(0, 0, 0, 0);
  if (tid == 0) {
    for (int s = 0; s <= kStages; ++s) mbar_init(&bars[s], 1);
    fence_mbar_init();
  }
  if (warp == 0) tc::alloc(tslot, kTmemCols);
  tc::fence_before();
  __syncthreads();
  tc::fence_after();
  const uint32_t tmem = *tslot;
  const int K64 = k64_tiles(p.d);
  const int nks = (K64 + 1) / 2;
  const int n_steps = n_units * nks;
  Loader ld;
  loader_init(p, ld, n_units);
  // prologue: stages 0 .. kStages-2
  for (int j = 0; j < kStages - 1; ++j) {
    loader_issue(p, ld, stages + (size_t)(j % kStages) * kStageBytes);
    cp_commit();
  }
  int unit_i = 0;
  TcUnit g = tc_unit(p, blockIdx.x);
  for (int j = 0; j < n_steps; ++j) {
    const int ks = j - unit_i * nks;
    // refill: stage j + kStages - 1 into the slot step j - 1 consumed (the threads copied it
    // out before the previous barrier; the tensor core reads only the operand buffers)
    const int jn = j + kStages - 1;
    if (jn < n_steps) loader_issue(p, ld, stages + (size_t)(jn % kStages) * kStageBytes);
    cp_commit();
    cp_wait<kStages - 1>();  // this thread's copies of stage j landed
    // the operand buffer and scale set of step j were last read by step j - 2's MMAs
    if (j >= 2) bounded_wait(&bars[(j - 2) & 1], (uint32_t)(((j - 2) >> 1) & 1), p.status);
    __syncthreads();
    const int b = j % kStages, ab = j & 1;
    uint8_t* sb = stages + (size_t)b * kStageBytes;
    uint8_t* sA = abuf + (size_t)ab * kAStage;
    uint8_t* sBo = bbuf + (size_t)ab * kBStage;
    const uint8_t* sSb = sb + kRaw + kBStage;
    const int npad = max(8, (g.n + 7) & ~7), N = 2 * npad;
    const int nkt = min(2, K64 - 2 * ks);
    {
      // weights of stage j: fragment order -> padded operand layout. Area tk = 2t + kts,
      // 16-byte chunk L (lane L = 4 gr + c of the fragment layout) holds for q = 2 bb + rr
      // codes 8c..8c+7 of block bb of tile row gr + 8 rr: M row 16 t + gr + 8 rr, row chunk
      // 4 kts + 2 bb + (c >> 1), bytes (c & 1) * 4
      const int L = tid & 31, gr = L >> 2, c = L & 3;
#pragma unroll
      for (int i = 0; i < 16 * 32 / kThr; ++i) {
        const int tk = (tid >> 5) + (kThr / 32) * i, t = tk >> 1, kts = tk & 1;
        if (kts >= nkt) continue;
        const uint4 v = *reinterpret_cast<const uint4*>(sb + tk * kTileBytes + 16 * L);
        const uint32_t vv[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          const int bb = q >> 1, rr = q & 1;
          *reinterpret_cast<uint32_t*>(sA + t * 2048 + kts * 512 + (rr * 8 + 2 * bb + (c >> 1)) * 128 + gr * 16 +
                                       (c & 1) * 4) = vv[q];
        }
      }
      // x planes of stage j -> operand buffer ab (rows of the unit's 2 npad B rows)
      for (int o = tid; o < npad * 2 * kStageK / 16; o += kThr)
        reinterpret_cast<uint4*>(sBo)[o] = reinterpret_cast<const uint4*>(sb + kRaw)[o];
      // scale factors of stage j -> TMEM set ab (warps 0..3, one per lane quadrant)
      if (warp < 4) {
      uint32_t wa[4];
#pragma unroll
      for (int r = 0; r < 4; ++r) {
        const int m = 32 * r + lane, t = m >> 4, rho = m & 15, g8 = rho & 7, rr = rho >> 3;
        uint32_t w = 0;
#pragma unroll
        for (int kb = 0; kb < 4; ++kb) {
          const int kts = kb >> 1, bb = kb & 1;
          w |= (uint32_t)sb[(t * 2 + kts) * kTileBytes + kTileCodeBytes + 4 * g8 + 2 * bb + rr] << (8 * kb);
        }
        wa[r] = w;
      }
      const uint32_t lanebase = tmem + ((uint32_t)(warp * 32) << 16) + kSfCol + 16 * ab;
      tc::st4(lanebase, wa[0], wa[1], wa[2], wa[3]);
      uint32_t wb[3];
#pragma unroll
      for (int r = 0; r < 3; ++r) {
        const int n = 32 * r + lane;
        wb[r] = n < N ? *reinterpret_cast<const uint32_t*>(sSb + 4 * n) : 0x7F7F7F7Fu;
      }
      tc::st4(lanebase + 8, wb[0], wb[1], wb[2], 0x7F7F7F7Fu);
      tc::wait_st();
      }
    }
    tc::fence_proxy_async();
    tc::fence_before();
    __syncthreads();
    const bool last = ks == nks - 1;
    if (tid == 0) {
      tc::fence_after();
      for (int kts = 0; kts < nkt; ++kts)
        for (int bb = 0; bb < 2; ++bb) {
          const int kb = 2 * kts + bb, kc = 4 * kts + 2 * bb;
          const uint64_t ad = tc::smem_desc(sA + kc * 128, 128, 8 * 128);
          const uint64_t bd = tc::smem_desc(sBo + kc * 128, 128, 8 * 128);
          tc::mma_mxf4_mxf8(tmem, ad, bd, tc::idesc_mxf4_mxf8(128, N, kb, kb), tmem + kSfCol + 16 * ab,
                            tmem + kSfCol + 16 * ab + 8, (ks > 0 || kb > 0) ? 1u : 0u);
        }
      tc::commit(&bars[ab]);
      if (last) tc::commit(&bars[kStages]);
    }
    if (!last) continue;
    // ---------------- epilogue of the unit: h = SiLU(gate) * up
    bounded_wait(&bars[kStages], (uint32_t)(unit_i & 1), p.status);
    tc::fence_after();
    // warp w reads lane quadrant qd = w & 3 and token columns [16 part, 16 part + 16), part = w >> 2
    const int qd = warp & 3, c0 = 16 * (warp >> 2);
    const uint32_t trow = tmem + ((uint32_t)(qd * 32) << 16);
    if (qd >= 2 && c0 < npad) {  // up rows 64 + 32 (qd - 2) + lane -> shared memory
      float hi[16], lo[16];
      tc::ld16(trow + c0, hi);
      tc::ld16(trow + npad + c0, lo);
#pragma unroll
      for (int i = 0; i < 16; ++i)
        if (c0 + i < g.n) upx[(32 * (qd - 2) + lane) * kMaxTok + c0 + i] = hi[i] + lo[i];
    }
    __syncthreads();
    if (qd < 2 && c0 < npad) {  // gate rows 32 qd + lane: pair tile tau0 + 2 qd + lane / 16, row lane % 16
      const int tau = g.tau0 + 2 * qd + (lane >> 4), r = lane & 15;
      const bool valid = tau < g.f / 16;
      {
        float hi[16], lo[16];
        tc::ld16(trow + c0, hi);
        tc::ld16(trow + npad + c0, lo);
#pragma unroll
        for (int i = 0; i < 16; ++i) {
          const int m = c0 + i;
          if (m >= g.n) break;  // uniform over the warp
          const float gate = hi[i] + lo[i];
          const float up = upx[(32 * qd + lane) * kMaxTok + m];
          const float h = gate / (1.f + expf(-gate)) * up;
          float mx = fabsf(h);
          for (int o = 1; o < 16; o <<= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
          if (valid) {
            const int q = g.q0 + m;
            const int sh = f16_headroom_exponent(mx);
            __half* hh = reinterpret_cast<__half*>(p.hbuf) + (size_t)q * 2 * p.fmax64;
            const int ii = 32 * (tau >> 1) + 8 * (r >> 2) + 4 * (tau & 1) + (r & 3);
            const float v = h * pow2f(sh);
            const __half vh = __float2half_rn(v);
            hh[ii] = vh;
            hh[p.fmax64 + ii] = __float2half_rn(v - __half2float(vh));
            if (r == 0) p.hscale[(size_t)q * p.hgroups + tau] = pow2f(-sh);
          }
        }
      }
    }
    tc::fence_before();
    __syncthreads();  // the accumulators and the up buffer are free for the next unit
    tc::fence_after();
    ++unit_i;
    if (unit_i < n_units) g = tc_unit(p, blockIdx.x + unit_i * gridDim.x);
  }
  cp_wait<0>();
  tc::fence_before();
  __syncthreads();
  if (warp == 0) tc::dealloc(tmem, kTmemCols);
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

constexpr size_t kTcSmem = (size_t)kStages * kStageBytes + 2 * (size_t)kAStage + 2 * (size_t)kBStage +
                           (size_t)64 * kMaxTok * 4 + 8 * (kStages + 1) + 16;

}  // namespace

cudaError_t launch_gemm_gateup_tc(const FwdParams& p, cudaStream_t stream, int num_sms) {
  static bool configured = false;
  if (!configured) {
    cudaError_t e = cudaFuncSetAttribute(gemm_gateup_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kTcSmem);
    if (e != cudaSuccess) return e;
    configured = true;
  }
  prep_xq_kernel<<<(p.T + 7) / 8, 256, 0, stream>>>(p);
  gemm_gateup_tc_kernel<<<num_sms, kThr, kTcSmem, stream>>>(p);
  return cudaGetLastError();
}

}  // namespace moe
