// Expert GEMMs of the general path (any T; the prefill chunk is its main
// user): gate/up + SwiGLU, then down, each over the work list of (slot,
// 12 weight tiles, block of up to 48 rows of the slot).
//
// A CTA (12 warps) takes one unit at a time; warp w owns weight tile w of the
// unit (a 16-row gate/up pair tile, or 16 down rows) over the whole reduction
// dimension, so no partial sums cross warps. Every warp streams its own
// tile's k tiles -- one contiguous range of the packed expert -- through a
// private shared-memory ring with cp.async. The activations of the unit's
// rows (x for gate/up, h for down) are staged for the whole CTA in chunks of
// k tiles, double-buffered: cp.async by all threads, completion on an
// mbarrier, one CTA barrier per chunk before its buffer is refilled. Both
// streams run on across unit boundaries.
//
// The math is the decode path's: MXFP4 codes decode exactly to f16 in
// registers (cvt.rn.f16x2.e2m1x2), m16n8k16 tensor-core MMAs with fp32
// accumulation, each 32-element block's E8M0 scale applied in fp32 to its
// partial sum; every output is one warp's fixed-order sum, so results do not
// depend on the batch or on timing.
//
// The pages: tokens grouped by expert on the GPU for the prompt, one GEMM per
// expert over its rows ("Neural Server" technical page, "Prompt processing");
// one pass over each selected expert's rows for all of its tokens ("NInfer"
// Qwen3.8-Flash-Next notes, MoE execution bullets).
#include <stdint.h>

#include "../../include/moe.h"
#include "moe_device.cuh"
#include "moe_internal.h"

namespace moe {
namespace {

using namespace dev;

constexpr int kGW = kGemmTiles;         // warps per CTA: one 16-row weight tile each
constexpr int kGThreads = kGW * 32;
constexpr int kRing = 6;                // per-warp weight ring slots of kGroup bytes
constexpr int kGroup = 2 * kTileBytes;  // a gate/up tile pair, or two down tiles
constexpr int kXC = 8;                  // k tiles per x chunk
constexpr int kHC = 4;                  // k tiles per h chunk
// Row strides of the staged activations: 64 bytes past a multiple of 128, so
// the 8 rows x 4 16-byte columns of a B-fragment load hit distinct banks.
constexpr int kXS = kXC * 64 + 32;      // f16 per row of an x chunk
constexpr int kHS = kHC * 64 + 32;      // f16 per (row, plane) of an h chunk

// A unit of either GEMM: slot, group of kGemmTiles weight tiles, block of rows.
struct GUnit {
  int e, f;      // expert (E = shared), its ffn
  int q0, n;     // first h/part row of the block and its rows (<= kGemmRows)
  int tile0;     // first weight tile (pair tile for gate/up, row tile for down)
};

__device__ __forceinline__ GUnit gemm_unit(const FwdParams& p, const int32_t* prefix, int u, bool down) {
  const int ns = *p.n_slots;
  const int s = find_unit_slot(prefix, ns, u);
  const int r = u - prefix[s];
  GUnit g;
  g.e = p.slot_expert[s];
  g.f = (g.e == p.E) ? p.S : p.F;
  const int tiles = down ? p.d / 16 : g.f / 16;
  const int ngrp = (tiles + kGW - 1) / kGW;
  const int tb = r / ngrp, grp = r - tb * ngrp;
  g.q0 = p.slot_q0[s] + kGemmRows * tb;
  g.n = min(kGemmRows, p.slot_n[s] - kGemmRows * tb);
  g.tile0 = kGW * grp;
  return g;
}

__device__ __forceinline__ int token_of_row(const FwdParams& p, int q) { return q < p.P ? p.perm[q] / p.k : q - p.P; }

// ---------------------------------------------------------------- gate/up

// Weight stream of one warp in the gate/up GEMM: its pair tile's K64(d) tile
// pairs in each of the CTA's units, one 1,088-byte ring slot per pair.
struct WStream {
  int i;             // CTA-local unit index of the next slot to issue
  int kt;            // k tile within that unit
  int n_units;
  const uint8_t* src;
  int left;          // slots left in the current unit
};

__device__ __forceinline__ void ws_seek_gu(const FwdParams& p, int w, WStream& ws) {
  const int K64 = k64_tiles(p.d);
  while (ws.i < ws.n_units) {
    const GUnit g = gemm_unit(p, p.gu_prefix, blockIdx.x + ws.i * gridDim.x, false);
    const int tau = g.tile0 + w;
    if (tau < g.f / 16) {
      ws.src = p.packed + (size_t)weight_index(p, g.e) * p.expert_stride + (size_t)tau * K64 * kGroup;
      ws.left = K64;
      return;
    }
    ++ws.i;
  }
}

__device__ __forceinline__ void ws_issue_gu(const FwdParams& p, int w, WStream& ws, uint8_t* dst) {
  const int lane = threadIdx.x & 31;
  if (ws.i < ws.n_units) {
    for (int k = lane; k < kGroup / 16; k += 32) cp16(dst + 16 * k, ws.src + 16 * k);
    ws.src += kGroup;
    if (--ws.left == 0) {
      ++ws.i;
      ws_seek_gu(p, w, ws);
    }
  }
  cp_commit();
}

// Stage x chunk j of the CTA's chunk sequence (unit j / nch, chunk j % nch)
// into buffer `xb`: rows m < n of the unit are the f16 x of its tokens.
__device__ __forceinline__ void load_x_chunk(const FwdParams& p, int j, int nch, __half* xb, uint64_t* bar) {
  const int i = j / nch, c = j - i * nch;
  const GUnit g = gemm_unit(p, p.gu_prefix, blockIdx.x + i * gridDim.x, false);
  const int k0 = c * kXC * 64, kw = min(kXC * 64, p.d64 - k0);
  const int per_row = kw / 8;
  for (int o = threadIdx.x; o < g.n * per_row; o += kGThreads) {
    const int m = o / per_row, k = o - m * per_row;
    const int t = token_of_row(p, g.q0 + m);
    cp16(xb + (size_t)m * kXS + 8 * k, p.x16 + (size_t)t * p.d64 + k0 + 8 * k);
  }
  cp_arrive(bar);
}

template <int NT>
__device__ void gemm_gu_unit(const FwdParams& p, const GUnit& g, int w, uint8_t* ring, int& slot, WStream& ws,
                             __half* xbuf, uint64_t* xbar, int& j, int nch, int n_chunks_total) {
  const int lane = threadIdx.x & 31, gq = lane >> 2, c = lane & 3;
  const int K64 = k64_tiles(p.d);
  const int tau = g.tile0 + w;
  const bool mine = tau < g.f / 16;
  float acc[2][NT][4];
#pragma unroll
  for (int h = 0; h < 2; ++h)
#pragma unroll
    for (int nt = 0; nt < NT; ++nt)
#pragma unroll
      for (int r = 0; r < 4; ++r) acc[h][nt][r] = 0.f;
  for (int ch = 0; ch < nch; ++ch, ++j) {
    const int b = j & 1;
    wait_chunk(&xbar[b], (uint32_t)((j >> 1) & 1), p.status);
    const __half* xc = xbuf + (size_t)b * kGemmRows * kXS;
    if (mine) {
      const int kt1 = min(K64, (ch + 1) * kXC);
      for (int kt = ch * kXC; kt < kt1; ++kt) {
        cp_wait<kRing - 1>();
        __syncwarp();
        const uint8_t* sl = ring + slot * kGroup;
        const int ktl = kt - ch * kXC;
        float scl[2][4];
        uint4 q[2];
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          q[h] = *reinterpret_cast<const uint4*>(sl + h * kTileBytes + 16 * lane);
          e8m0x4_f32(*reinterpret_cast<const uint32_t*>(sl + h * kTileBytes + kTileCodeBytes + 4 * gq), scl[h]);
        }
#pragma unroll
        for (int bb = 0; bb < 2; ++bb)
#pragma unroll
          for (int h = 0; h < 2; ++h) {
            uint32_t a1[4], a2[4];
            a_frags(q[h], bb, a1, a2);
            const float sg = scl[h][2 * bb], sg8 = scl[h][2 * bb + 1];
#pragma unroll
            for (int nt = 0; nt < NT; ++nt) {
              const uint4 bx =
                  *reinterpret_cast<const uint4*>(xc + (size_t)(8 * nt + gq) * kXS + ktl * 64 + bb * 32 + c * 8);
              float t[4];
              mma_z(t, a1, bx.x, bx.y);
              mma16816(t, a2, bx.z, bx.w);
              acc[h][nt][0] = fmaf(t[0], sg, acc[h][nt][0]);
              acc[h][nt][1] = fmaf(t[1], sg, acc[h][nt][1]);
              acc[h][nt][2] = fmaf(t[2], sg8, acc[h][nt][2]);
              acc[h][nt][3] = fmaf(t[3], sg8, acc[h][nt][3]);
            }
          }
        __syncwarp();
        ws_issue_gu(p, w, ws, ring + slot * kGroup);
        if (++slot == kRing) slot = 0;
      }
    }
    __syncthreads();  // every warp is done with buffer b
    if (j + 2 < n_chunks_total) load_x_chunk(p, j + 2, nch, xbuf + (size_t)b * kGemmRows * kXS, &xbar[b]);
  }
  if (!mine) return;
  // SwiGLU epilogue: rows S_tau (g, g + 8) of columns 8 nt + 2c (+1)
#pragma unroll
  for (int nt = 0; nt < NT; ++nt) {
    float hv[4];
#pragma unroll
    for (int r = 0; r < 4; ++r) {
      const int m = 8 * nt + 2 * c + (r & 1);
      float h = 0.f;
      if (m < g.n) {
        const float xi = p.xinv[token_of_row(p, g.q0 + m)];
        const float gate = acc[0][nt][r] * xi, up = acc[1][nt][r] * xi;
        h = gate / (1.f + expf(-gate)) * up;
      }
      hv[r] = h;
    }
    float mx0 = fmaxf(fabsf(hv[0]), fabsf(hv[2]));
    float mx1 = fmaxf(fabsf(hv[1]), fabsf(hv[3]));
    for (int o = 4; o < 32; o <<= 1) {
      mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, o));
      mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, o));
    }
#pragma unroll
    for (int col = 0; col < 2; ++col) {
      const int m = 8 * nt + 2 * c + col;
      if (m >= g.n) continue;
      const int q = g.q0 + m;
      const int sh = f16_headroom_exponent(col ? mx1 : mx0);
      const float sc = pow2f(sh);
      __half* hi = reinterpret_cast<__half*>(p.hbuf) + (size_t)q * 2 * p.fmax64;
      __half* lo = hi + p.fmax64;
#pragma unroll
      for (int half = 0; half < 2; ++half) {
        const int rr = gq + 8 * half;
        const int i = 32 * (tau >> 1) + 8 * (rr >> 2) + 4 * (tau & 1) + (rr & 3);
        const float v = hv[2 * half + col] * sc;
        const __half vh = __float2half_rn(v);
        hi[i] = vh;
        lo[i] = __float2half_rn(v - __half2float(vh));
      }
      if (gq == 0) p.hscale[(size_t)q * p.hgroups + tau] = pow2f(-sh);
    }
  }
}

__global__ void __launch_bounds__(kGThreads, 1) gemm_gateup_kernel(FwdParams p) {
  pdl_enter();
  extern __shared__ __align__(128) uint8_t sm[];
  uint64_t* xbar = reinterpret_cast<uint64_t*>(sm);
  __half* xbuf = reinterpret_cast<__half*>(sm + 128);
  uint8_t* rings = sm + 128 + (size_t)2 * kGemmRows * kXS * 2;
  const int w = threadIdx.x >> 5;
  const int total = p.gu_prefix[*p.n_slots];
  const int n_units = total > (int)blockIdx.x ? (total - (int)blockIdx.x + gridDim.x - 1) / gridDim.x : 0;
  if (n_units == 0) return;
  if (threadIdx.x == 0) {
    mbar_init(&xbar[0], kGThreads);
    mbar_init(&xbar[1], kGThreads);
    fence_mbar_init();
  }
  __syncthreads();
  const int nch = (k64_tiles(p.d) + kXC - 1) / kXC;
  const int n_chunks_total = n_units * nch;
  load_x_chunk(p, 0, nch, xbuf, &xbar[0]);
  if (n_chunks_total > 1) load_x_chunk(p, 1, nch, xbuf + (size_t)kGemmRows * kXS, &xbar[1]);
  uint8_t* ring = rings + (size_t)w * kRing * kGroup;
  WStream ws;
  ws.i = 0;
  ws.n_units = n_units;
  ws_seek_gu(p, w, ws);
  for (int s = 0; s < kRing; ++s) ws_issue_gu(p, w, ws, ring + s * kGroup);
  int slot = 0, j = 0;
  for (int i = 0; i < n_units; ++i) {
    const GUnit g = gemm_unit(p, p.gu_prefix, blockIdx.x + i * gridDim.x, false);
    const int nt = (g.n + 7) / 8;
    switch (nt) {
      case 1: gemm_gu_unit<1>(p, g, w, ring, slot, ws, xbuf, xbar, j, nch, n_chunks_total); break;
      case 2: gemm_gu_unit<2>(p, g, w, ring, slot, ws, xbuf, xbar, j, nch, n_chunks_total); break;
      case 3: gemm_gu_unit<3>(p, g, w, ring, slot, ws, xbuf, xbar, j, nch, n_chunks_total); break;
      case 4: gemm_gu_unit<4>(p, g, w, ring, slot, ws, xbuf, xbar, j, nch, n_chunks_total); break;
      case 5: gemm_gu_unit<5>(p, g, w, ring, slot, ws, xbuf, xbar, j, nch, n_chunks_total); break;
      default: gemm_gu_unit<6>(p, g, w, ring, slot, ws, xbuf, xbar, j, nch, n_chunks_total); break;
    }
  }
  cp_wait_all();
}

// ---------------------------------------------------------------- down

__device__ __forceinline__ void ws_seek_dn(const FwdParams& p, int w, WStream& ws) {
  while (ws.i < ws.n_units) {
    const GUnit g = gemm_unit(p, p.dn_prefix, blockIdx.x + ws.i * gridDim.x, true);
    const int m = g.tile0 + w;
    if (m < p.d / 16) {
      const int K64 = k64_tiles(g.f);
      ws.src = p.packed + (size_t)weight_index(p, g.e) * p.expert_stride + gu_packed_bytes(p.d, g.f) +
               (size_t)m * K64 * kTileBytes;
      ws.kt = 0;
      ws.left = K64;  // tiles
      return;
    }
    ++ws.i;
  }
}

// One slot of the down stream: the next two k tiles of the warp's row tile
// (one at the end of an odd K64(f)).
__device__ __forceinline__ void ws_issue_dn(const FwdParams& p, int w, WStream& ws, uint8_t* dst) {
  const int lane = threadIdx.x & 31;
  if (ws.i < ws.n_units) {
    const int nt = min(2, ws.left);
    for (int k = lane; k < nt * kTileBytes / 16; k += 32) cp16(dst + 16 * k, ws.src + 16 * k);
    ws.src += nt * kTileBytes;
    ws.left -= nt;
    if (ws.left == 0) {
      ++ws.i;
      ws_seek_dn(p, w, ws);
    }
  }
  cp_commit();
}

// The down GEMM's chunk sequence: the CTA's units of routed slots come
// first (nch0 chunks each), those of the shared expert last (nch1 each).
struct ChunkMap {
  int n_first, nch0, nch1;
};

__device__ __forceinline__ void chunk_unit(const ChunkMap& cm, int j, int& i, int& c) {
  if (j < cm.n_first * cm.nch0) {
    i = j / cm.nch0;
    c = j - i * cm.nch0;
  } else {
    const int r = j - cm.n_first * cm.nch0;
    i = cm.n_first + r / cm.nch1;
    c = r - (i - cm.n_first) * cm.nch1;
  }
}

// Stage h chunk j: for rows m < n of its unit, both f16 planes of k tiles
// [kHC c, kHC c + kHC) and their scales.
__device__ __forceinline__ void load_h_chunk(const FwdParams& p, int j, const ChunkMap& cm, __half* hb, float* hs,
                                             uint64_t* bar) {
  int i, c;
  chunk_unit(cm, j, i, c);
  const GUnit g = gemm_unit(p, p.dn_prefix, blockIdx.x + i * gridDim.x, true);
  const int k0 = c * kHC * 64, kw = min(kHC * 64, k64_tiles(g.f) * 64 - k0);
  const int per_plane = kw / 8;
  for (int o = threadIdx.x; o < g.n * 2 * per_plane; o += kGThreads) {
    const int mp = o / per_plane, k = o - mp * per_plane;  // mp = 2 m + plane
    cp16(hb + (size_t)mp * kHS + 8 * k, p.hbuf + ((size_t)(g.q0 + (mp >> 1)) * 2 + (mp & 1)) * p.fmax64 + k0 + 8 * k);
  }
  const int per_row = kw / 64;  // 16-byte pieces of scales: 4 per k tile
  for (int o = threadIdx.x; o < g.n * per_row; o += kGThreads) {
    const int m = o / per_row, k = o - m * per_row;
    cp16(hs + (size_t)m * kHC * 4 + 4 * k, p.hscale + (size_t)(g.q0 + m) * p.hgroups + c * kHC * 4 + 4 * k);
  }
  cp_arrive(bar);
}

template <int NT>
__device__ void gemm_dn_unit(const FwdParams& p, const GUnit& g, int w, uint8_t* ring, int& slot, WStream& ws,
                             __half* hbuf, float* hsbuf, uint64_t* hbar, int& j, const ChunkMap& cm,
                             int n_chunks_total) {
  const int nch = (k64_tiles(g.f) + kHC - 1) / kHC;
  const int lane = threadIdx.x & 31, gq = lane >> 2, c = lane & 3;
  const int K64 = k64_tiles(g.f);
  const int m = g.tile0 + w;
  const bool mine = m < p.d / 16;
  float acc[NT][2];
#pragma unroll
  for (int nt = 0; nt < NT; ++nt) acc[nt][0] = acc[nt][1] = 0.f;
  int in_slot = 0;  // tiles of the current ring slot already used
  for (int ch = 0; ch < nch; ++ch, ++j) {
    const int b = j & 1;
    wait_chunk(&hbar[b], (uint32_t)((j >> 1) & 1), p.status);
    const __half* hc = hbuf + (size_t)b * kGemmRows * 2 * kHS;
    const float* sc4 = hsbuf + (size_t)b * kGemmRows * kHC * 4;
    if (mine) {
      const int kt1 = min(K64, (ch + 1) * kHC);
      for (int kt = ch * kHC; kt < kt1; ++kt) {
        if (in_slot == 0) {
          cp_wait<kRing - 1>();
          __syncwarp();
        }
        const uint8_t* t8 = ring + slot * kGroup + in_slot * kTileBytes;
        const int ktl = kt - ch * kHC;
        const uint4 q = *reinterpret_cast<const uint4*>(t8 + 16 * lane);
        float scl[4];
        e8m0x4_f32(*reinterpret_cast<const uint32_t*>(t8 + kTileCodeBytes + 4 * gq), scl);
#pragma unroll
        for (int bb = 0; bb < 2; ++bb) {
          uint32_t a1[4], a2[4];
          a_frags(q, bb, a1, a2);
          const float sg = scl[2 * bb], sg8 = scl[2 * bb + 1];
#pragma unroll
          for (int nt = 0; nt < NT; ++nt) {
            const uint4 bh = *reinterpret_cast<const uint4*>(hc + (size_t)((4 * nt + (gq >> 1)) * 2 + (gq & 1)) * kHS +
                                                             ktl * 64 + bb * 32 + c * 8);
            const float2 s2 = *reinterpret_cast<const float2*>(sc4 + (size_t)(4 * nt + c) * kHC * 4 + 2 * (2 * ktl + bb));
            float t1[4], t2[4];
            mma_z(t1, a1, bh.x, bh.y);
            mma_z(t2, a2, bh.z, bh.w);
            acc[nt][0] = fmaf(t1[0] + t1[1], sg * s2.x, acc[nt][0]);
            acc[nt][0] = fmaf(t2[0] + t2[1], sg * s2.y, acc[nt][0]);
            acc[nt][1] = fmaf(t1[2] + t1[3], sg8 * s2.x, acc[nt][1]);
            acc[nt][1] = fmaf(t2[2] + t2[3], sg8 * s2.y, acc[nt][1]);
          }
        }
        if (++in_slot == 2 || kt + 1 == K64) {
          in_slot = 0;
          __syncwarp();
          ws_issue_dn(p, w, ws, ring + slot * kGroup);
          if (++slot == kRing) slot = 0;
        }
      }
    }
    __syncthreads();  // every warp is done with buffer b
    if (j + 2 < n_chunks_total)
      load_h_chunk(p, j + 2, cm, hbuf + (size_t)b * kGemmRows * 2 * kHS, hsbuf + (size_t)b * kGemmRows * kHC * 4,
                   &hbar[b]);
  }
  if (!mine) return;
#pragma unroll
  for (int nt = 0; nt < NT; ++nt) {
    const int md = 4 * nt + c;
    if (md < g.n) {
      float* dst = p.part + (size_t)(g.q0 + md) * p.d + 16 * m;
      dst[gq] = acc[nt][0];
      dst[gq + 8] = acc[nt][1];
    }
  }
}

__global__ void __launch_bounds__(kGThreads, 1) gemm_down_kernel(FwdParams p) {
  pdl_enter();
  extern __shared__ __align__(128) uint8_t sm[];
  uint64_t* hbar = reinterpret_cast<uint64_t*>(sm);
  __half* hbuf = reinterpret_cast<__half*>(sm + 128);
  float* hsbuf = reinterpret_cast<float*>(sm + 128 + (size_t)2 * kGemmRows * 2 * kHS * 2);
  uint8_t* rings = reinterpret_cast<uint8_t*>(hsbuf + (size_t)2 * kGemmRows * kHC * 4);
  const int w = threadIdx.x >> 5;
  const int total = p.dn_prefix[*p.n_slots];
  const int n_units = total > (int)blockIdx.x ? (total - (int)blockIdx.x + gridDim.x - 1) / gridDim.x : 0;
  if (n_units == 0) return;
  if (threadIdx.x == 0) {
    mbar_init(&hbar[0], kGThreads);
    mbar_init(&hbar[1], kGThreads);
    fence_mbar_init();
  }
  __syncthreads();
  ChunkMap cm;
  cm.nch0 = (k64_tiles(p.F) + kHC - 1) / kHC;
  cm.nch1 = p.S > 0 ? (k64_tiles(p.S) + kHC - 1) / kHC : cm.nch0;
  const int ns = *p.n_slots;
  // first unit of the shared expert (its slot is last, on the shard with e_begin == 0 only)
  const int split = (p.S > 0 && p.e_begin == 0) ? p.dn_prefix[ns - 1] : total;
  cm.n_first = split > (int)blockIdx.x ? min(n_units, (split - (int)blockIdx.x + gridDim.x - 1) / gridDim.x) : 0;
  const int n_chunks_total = cm.n_first * cm.nch0 + (n_units - cm.n_first) * cm.nch1;
  load_h_chunk(p, 0, cm, hbuf, hsbuf, &hbar[0]);
  if (n_chunks_total > 1)
    load_h_chunk(p, 1, cm, hbuf + (size_t)kGemmRows * 2 * kHS, hsbuf + (size_t)kGemmRows * kHC * 4, &hbar[1]);
  uint8_t* ring = rings + (size_t)w * kRing * kGroup;
  WStream ws;
  ws.i = 0;
  ws.n_units = n_units;
  ws_seek_dn(p, w, ws);
  for (int s = 0; s < kRing; ++s) ws_issue_dn(p, w, ws, ring + s * kGroup);
  int slot = 0, j = 0;
  for (int i = 0; i < n_units; ++i) {
    const GUnit g = gemm_unit(p, p.dn_prefix, blockIdx.x + i * gridDim.x, true);
    const int nt = (g.n + 3) / 4;  // 4 rows (hi and lo columns) per n8 tile
    if (nt <= 2) gemm_dn_unit<2>(p, g, w, ring, slot, ws, hbuf, hsbuf, hbar, j, cm, n_chunks_total);
    else if (nt <= 4) gemm_dn_unit<4>(p, g, w, ring, slot, ws, hbuf, hsbuf, hbar, j, cm, n_chunks_total);
    else if (nt <= 6) gemm_dn_unit<6>(p, g, w, ring, slot, ws, hbuf, hsbuf, hbar, j, cm, n_chunks_total);
    else if (nt <= 8) gemm_dn_unit<8>(p, g, w, ring, slot, ws, hbuf, hsbuf, hbar, j, cm, n_chunks_total);
    else if (nt <= 10) gemm_dn_unit<10>(p, g, w, ring, slot, ws, hbuf, hsbuf, hbar, j, cm, n_chunks_total);
    else gemm_dn_unit<12>(p, g, w, ring, slot, ws, hbuf, hsbuf, hbar, j, cm, n_chunks_total);
  }
  cp_wait_all();
}

constexpr size_t kGuSmem = 128 + (size_t)2 * kGemmRows * kXS * 2 + (size_t)kGW * kRing * kGroup;
constexpr size_t kDnSmem =
    128 + (size_t)2 * kGemmRows * 2 * kHS * 2 + (size_t)2 * kGemmRows * kHC * 4 * 4 + (size_t)kGW * kRing * kGroup;

}  // namespace

cudaError_t configure_gemm() {
  cudaError_t e = cudaFuncSetAttribute(gemm_gateup_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kGuSmem);
  if (e == cudaSuccess)
    e = cudaFuncSetAttribute(gemm_down_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kDnSmem);
  return e;
}

cudaError_t launch_gemm_gateup(const FwdParams& p, cudaStream_t stream, int num_sms) {
  gemm_gateup_kernel<<<num_sms, kGThreads, kGuSmem, stream>>>(p);
  return cudaGetLastError();
}

cudaError_t launch_gemm_down(const FwdParams& p, cudaStream_t stream, int num_sms) {
  gemm_down_kernel<<<num_sms, kGThreads, kDnSmem, stream>>>(p);
  return cudaGetLastError();
}

}  // namespace moe
