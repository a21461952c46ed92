// Expert GEMMs of the general path for affine group-64 experts: gate/up +
// SwiGLU, then down, with w = scale * q + bias (q a `bits`-bit unsigned code,
// one bf16 scale and one bf16 bias per 64 weights of a row).
//
// The pages keep their routed experts in this form ("Running
// Qwen3.8-Flash-Next on a 32 GB Mac with Transformers": the table of where
// every weight lives -- 3-bit affine, group 64, a 16-bit scale and bias per 64
// weights, 2.15 MB per expert) and decode them in registers inside the GEMV of
// the CUDA port (same page, "CUDA (preview)": the kernel that unpacks the
// format in registers).
//
// Per group the dot product splits exactly into
//   sum_c (s q_c + b) x_c = s * sum_c q_c x_c + b * sum_c x_c,
// so the tensor cores only see the integer codes. A lane turns two codes into
// one A register with a shift and a mask: the f16 with exponent field 0 and
// mantissa q is the subnormal q * 2^-24, exact, so the m16n8k16 MMA (f16
// inputs, fp32 accumulation) yields 2^-24 sum_c q_c x_c over the group's 64
// columns (four k16 MMAs into a fresh accumulator), and the warp adds
// (s 2^24) * that + b * sum_c x_c to its running fp32 sum. The activations
// are the f16 planes the register-decode path already uses: x * 2^sigma_t
// (one f16 per element) for gate/up, and h as two f16 planes with a scale
// 2^-sh per 16 elements for down; the group sums of both come with them.
//
// Work: one warp per item (slot, one 16-row weight tile, block of up to
// kAffRows rows of the slot); the item's weight tiles stream through the
// warp's own cp.async ring in shared memory and the warp continues into its
// next item without a CTA barrier. Activation fragments are read through L1
// (a slot's few rows of x or h are shared by the warps of its items). Every
// output is one warp's sum in a fixed order, so results do not depend on the
// batch or on timing.
#include <stdint.h>

#include "../../include/moe.h"
#include "moe_device.cuh"
#include "moe_internal.h"

namespace moe {
namespace {

using namespace dev;

constexpr int kAW = 8;                   // warps per CTA
constexpr int kAThreads = kAW * 32;
constexpr int kARingBytes = 11 * 1024;   // per-warp weight ring
constexpr size_t kASmem = (size_t)kAW * kARingBytes;

template <int B>
struct Aff {
  static constexpr int kTile = 128 * B + 64;
  static constexpr int kSlot = 2 * kTile;  // a gate/up tile pair, or two down tiles
  static constexpr int kRing = kARingBytes / kSlot;
  static_assert(kRing >= 2, "ring too shallow");
};

// Codes of pair p of a lane's words (see aff_tile_bytes): the first code in
// bits [0, B), the second in bits [16, 16 + B) -- the f16 pair (q0, q1) 2^-24.
template <int B, int P>
__device__ __forceinline__ uint32_t aff_pair(const uint32_t (&w)[B]) {
  constexpr int o = B * P, j = o >> 4, s = o & 15;
  constexpr uint32_t m = (1u << B) - 1u;
  if constexpr (s + B <= 16) {
    return (w[j] >> s) & (m * 0x00010001u);
  } else {
    constexpr int lo = 16 - s;  // bits of the field in word j
    constexpr uint32_t m_lo = (1u << lo) - 1u, m_hi = m ^ m_lo;
    return ((w[j] >> s) & (m_lo * 0x00010001u)) | ((w[j + 1] << lo) & (m_hi * 0x00010001u));
  }
}

template <int B, int KB>
__device__ __forceinline__ void aff_frag(const uint32_t (&w)[B], uint32_t (&a)[4]) {
  a[0] = aff_pair<B, 4 * KB + 0>(w);
  a[1] = aff_pair<B, 4 * KB + 1>(w);
  a[2] = aff_pair<B, 4 * KB + 2>(w);
  a[3] = aff_pair<B, 4 * KB + 3>(w);
}

__device__ __forceinline__ float bf16_lo(uint32_t v) { return __uint_as_float(v << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t v) { return __uint_as_float(v & 0xFFFF0000u); }
__device__ __forceinline__ uint2 ld8(const void* p) { return __ldg(reinterpret_cast<const uint2*>(p)); }

__device__ __forceinline__ int token_of_row(const FwdParams& p, int q) { return q < p.P ? p.perm[q] / p.k : q - p.P; }

struct AItem {
  int e, f;   // expert (E = shared) and its ffn
  int q0, n;  // first h/part row of the block and its rows (<= kAffRows)
  int tile;   // pair tile (gate/up) or row tile (down)
};

__device__ __forceinline__ AItem aff_item(const FwdParams& p, const int32_t* prefix, int u, bool down) {
  const int s = find_unit_slot(prefix, *p.n_slots, u);
  const int r = u - prefix[s];
  AItem it;
  it.e = p.slot_expert[s];
  it.f = it.e == p.E ? p.S : p.F;
  const int tiles = down ? p.d / 16 : it.f / 16;
  const int blk = r / tiles;
  it.tile = r - blk * tiles;
  it.q0 = p.slot_q0[s] + kAffRows * blk;
  it.n = min(kAffRows, p.slot_n[s] - kAffRows * blk);
  return it;
}

// The weight stream of one warp: the tiles of its items in order, two per ring
// slot (gate/up: the gate and up tiles of one k tile; down: two k tiles of the
// row tile, one at the end of an odd count).
struct AStream {
  int i, n_items, gw, nw;  // warp-local index of the item being issued, item count, first item, stride
  const uint8_t* src;
  int left;                // tiles of that item still to issue
};

template <int B>
__device__ __forceinline__ void aff_seek(const FwdParams& p, AStream& ws, bool down) {
  if (ws.i >= ws.n_items) return;
  const AItem it = aff_item(p, down ? p.dn_prefix : p.gu_prefix, ws.gw + ws.i * ws.nw, down);
  const uint8_t* base = p.packed + (size_t)weight_index(p, it.e) * p.expert_stride;
  if (down) {
    ws.src = base + aff_gu_bytes(p.d, it.f, B) + (size_t)it.tile * (it.f / 64) * Aff<B>::kTile;
    ws.left = it.f / 64;
  } else {
    ws.src = base + (size_t)it.tile * (p.d / 64) * Aff<B>::kSlot;
    ws.left = 2 * (p.d / 64);
  }
}

template <int B>
__device__ __forceinline__ void aff_issue(const FwdParams& p, AStream& ws, uint8_t* dst, bool down) {
  const int lane = threadIdx.x & 31;
  if (ws.i < ws.n_items) {
    const int nt = min(2, ws.left);
    for (int k = lane; k < nt * Aff<B>::kTile / 16; k += 32) cp16(dst + 16 * k, ws.src + 16 * k);
    ws.src += nt * Aff<B>::kTile;
    ws.left -= nt;
    if (ws.left == 0) {
      ++ws.i;
      aff_seek<B>(p, ws, down);
    }
  }
  cp_commit();
}

template <int B>
__device__ __forceinline__ void load_tile(const uint8_t* tile, int lane, uint32_t (&w)[B], uint2& sb) {
#pragma unroll
  for (int j = 0; j < B; ++j) w[j] = *reinterpret_cast<const uint32_t*>(tile + 4 * (B * lane + j));
  sb = *reinterpret_cast<const uint2*>(tile + 128 * B + 8 * (lane >> 2));
}

// ---------------------------------------------------------------- gate/up

template <int B, int NT>
__device__ void aff_gu_item(const FwdParams& p, const AItem& it, uint8_t* ring, int& slot, AStream& ws) {
  const int lane = threadIdx.x & 31, gq = lane >> 2, c = lane & 3;
  const int K64 = p.d / 64;
  int xo[NT];     // B fragment row 8 nt + gq: its token's x16 row offset, or -1 past the block
  int so[NT][2];  // C fragment column 8 nt + 2c + j: its token, or -1
#pragma unroll
  for (int nt = 0; nt < NT; ++nt) {
    const int m = 8 * nt + gq;
    xo[nt] = m < it.n ? token_of_row(p, it.q0 + m) * p.d64 : -1;
#pragma unroll
    for (int j = 0; j < 2; ++j) {
      const int mc = 8 * nt + 2 * c + j;
      so[nt][j] = mc < it.n ? token_of_row(p, it.q0 + mc) : -1;
    }
  }
  float acc[2][NT][4];
#pragma unroll
  for (int h = 0; h < 2; ++h)
#pragma unroll
    for (int nt = 0; nt < NT; ++nt)
#pragma unroll
      for (int r = 0; r < 4; ++r) acc[h][nt][r] = 0.f;
  const uint16_t* x16 = p.x16;
  for (int kt = 0; kt < K64; ++kt) {
    cp_wait<Aff<B>::kRing - 1>();
    __syncwarp();
    uint32_t w[2][B];
    uint2 sb[2];
    const uint8_t* sl = ring + slot * Aff<B>::kSlot;
    load_tile<B>(sl, lane, w[0], sb[0]);
    load_tile<B>(sl + Aff<B>::kTile, lane, w[1], sb[1]);
    __syncwarp();
    aff_issue<B>(p, ws, ring + slot * Aff<B>::kSlot, false);
    if (++slot == Aff<B>::kRing) slot = 0;
    float t[2][NT][4];
    uint2 bx[NT];
#define AFF_GU_KB(KB)                                                                                   \
  {                                                                                                    \
    uint32_t a0[4], a1[4];                                                                             \
    aff_frag<B, KB>(w[0], a0);                                                                         \
    aff_frag<B, KB>(w[1], a1);                                                                         \
    _Pragma("unroll") for (int nt = 0; nt < NT; ++nt) bx[nt] =                                          \
        xo[nt] >= 0 ? ld8(x16 + xo[nt] + 64 * kt + 16 * KB + 4 * c) : make_uint2(0u, 0u);              \
    _Pragma("unroll") for (int nt = 0; nt < NT; ++nt) {                                                 \
      if (KB == 0) {                                                                                   \
        mma_z(t[0][nt], a0, bx[nt].x, bx[nt].y);                                                       \
        mma_z(t[1][nt], a1, bx[nt].x, bx[nt].y);                                                       \
      } else {                                                                                         \
        mma16816(t[0][nt], a0, bx[nt].x, bx[nt].y);                                                    \
        mma16816(t[1][nt], a1, bx[nt].x, bx[nt].y);                                                    \
      }                                                                                                \
    }                                                                                                  \
  }
    AFF_GU_KB(0)
    AFF_GU_KB(1)
    AFF_GU_KB(2)
    AFF_GU_KB(3)
#undef AFF_GU_KB
    // the group's affine terms: rows gq (C registers 0, 1) and gq + 8 (2, 3)
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) {
      const float xs0 = so[nt][0] >= 0 ? p.xgsum[(size_t)so[nt][0] * p.xg_pitch + kt] : 0.f;
      const float xs1 = so[nt][1] >= 0 ? p.xgsum[(size_t)so[nt][1] * p.xg_pitch + kt] : 0.f;
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        const float s0 = bf16_lo(sb[h].x) * 0x1p24f, s1 = bf16_hi(sb[h].x) * 0x1p24f;
        const float b0 = bf16_lo(sb[h].y), b1 = bf16_hi(sb[h].y);
        acc[h][nt][0] = fmaf(s0, t[h][nt][0], fmaf(b0, xs0, acc[h][nt][0]));
        acc[h][nt][1] = fmaf(s0, t[h][nt][1], fmaf(b0, xs1, acc[h][nt][1]));
        acc[h][nt][2] = fmaf(s1, t[h][nt][2], fmaf(b1, xs0, acc[h][nt][2]));
        acc[h][nt][3] = fmaf(s1, t[h][nt][3], fmaf(b1, xs1, acc[h][nt][3]));
      }
    }
  }
  // SwiGLU epilogue: h rows 16 tau + gq (+ 8) of the block's rows 8 nt + 2c (+ 1),
  // stored as the down GEMM reads them (two f16 planes, a 2^-sh scale and the
  // group sum per 16 elements)
  const int tau = it.tile;
#pragma unroll
  for (int nt = 0; nt < NT; ++nt) {
#pragma unroll
    for (int col = 0; col < 2; ++col) {
      const int m = 8 * nt + 2 * c + col;
      const bool ok = m < it.n;
      const float xi = ok ? p.xinv[so[nt][col]] : 0.f;
      float hv[2];
#pragma unroll
      for (int r = 0; r < 2; ++r) {
        const float gate = acc[0][nt][2 * r + col] * xi, up = acc[1][nt][2 * r + col] * xi;
        hv[r] = ok ? gate / (1.f + expf(-gate)) * up : 0.f;
      }
      float mx = fmaxf(fabsf(hv[0]), fabsf(hv[1]));
#pragma unroll
      for (int o = 4; o < 32; o <<= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
      const int sh = f16_headroom_exponent(mx);
      const float sc = pow2f(sh);
      __half* hi = reinterpret_cast<__half*>(p.hbuf) + (size_t)(it.q0 + m) * 2 * p.fmax64;
      float rep = 0.f;
#pragma unroll
      for (int r = 0; r < 2; ++r) {
        const float v = hv[r] * sc;
        const __half vh = __float2half_rn(v);
        const __half vl = __float2half_rn(v - __half2float(vh));
        rep += __half2float(vh) + __half2float(vl);
        if (ok) {
          hi[16 * tau + gq + 8 * r] = vh;
          hi[p.fmax64 + 16 * tau + gq + 8 * r] = vl;
        }
      }
#pragma unroll
      for (int o = 4; o < 32; o <<= 1) rep += __shfl_xor_sync(0xffffffffu, rep, o);
      if (ok && gq == 0) {
        const size_t q = (size_t)(it.q0 + m) * p.hgroups + tau;
        p.hscale[q] = pow2f(-sh);
        p.hbsum[q] = rep * pow2f(-sh);
      }
    }
  }
}

template <int B>
__global__ void __launch_bounds__(kAThreads, 2) aff_gateup_kernel(FwdParams p) {
  pdl_enter();
  extern __shared__ __align__(128) uint8_t sm[];
  const int w = threadIdx.x >> 5;
  AStream ws;
  ws.gw = blockIdx.x * kAW + w;
  ws.nw = gridDim.x * kAW;
  const int total = p.gu_prefix[*p.n_slots];
  ws.n_items = total > ws.gw ? (total - ws.gw + ws.nw - 1) / ws.nw : 0;
  if (ws.n_items == 0) return;  // no CTA-wide barrier follows: warps are independent
  ws.i = 0;
  aff_seek<B>(p, ws, false);
  uint8_t* ring = sm + (size_t)w * kARingBytes;
  for (int s = 0; s < Aff<B>::kRing; ++s) aff_issue<B>(p, ws, ring + s * Aff<B>::kSlot, false);
  int slot = 0;
  for (int i = 0; i < ws.n_items; ++i) {
    const AItem it = aff_item(p, p.gu_prefix, ws.gw + i * ws.nw, false);
    const int nt = (it.n + 7) / 8;
    if (nt <= 1) aff_gu_item<B, 1>(p, it, ring, slot, ws);
    else if (nt <= 2) aff_gu_item<B, 2>(p, it, ring, slot, ws);
    else aff_gu_item<B, 4>(p, it, ring, slot, ws);
  }
  cp_wait_all();
}

// ---------------------------------------------------------------- down

template <int B, int NT>
__device__ void aff_dn_item(const FwdParams& p, const AItem& it, uint8_t* ring, int& slot, AStream& ws) {
  const int lane = threadIdx.x & 31, gq = lane >> 2, c = lane & 3;
  const int K64 = it.f / 64;
  int ho[NT];  // B fragment row gq of n8 tile nt = (block row 4 nt + gq / 2, plane gq % 2): hbuf offset, or -1
  int so[NT];  // C fragment columns 2c, 2c + 1 = both planes of block row 4 nt + c: its hscale row, or -1
#pragma unroll
  for (int nt = 0; nt < NT; ++nt) {
    const int r = 4 * nt + (gq >> 1), rc = 4 * nt + c;
    ho[nt] = r < it.n ? ((it.q0 + r) * 2 + (gq & 1)) * p.fmax64 : -1;
    so[nt] = rc < it.n ? (it.q0 + rc) * p.hgroups : -1;
  }
  float acc[NT][2];
#pragma unroll
  for (int nt = 0; nt < NT; ++nt) acc[nt][0] = acc[nt][1] = 0.f;
  const uint16_t* hb = p.hbuf;
  int in_slot = 0;
  for (int kt = 0; kt < K64; ++kt) {
    if (in_slot == 0) {
      cp_wait<Aff<B>::kRing - 1>();
      __syncwarp();
    }
    uint32_t w[B];
    uint2 sb;
    load_tile<B>(ring + slot * Aff<B>::kSlot + in_slot * Aff<B>::kTile, lane, w, sb);
    if (++in_slot == 2 || kt + 1 == K64) {
      in_slot = 0;
      __syncwarp();
      aff_issue<B>(p, ws, ring + slot * Aff<B>::kSlot, true);
      if (++slot == Aff<B>::kRing) slot = 0;
    }
    float gp[NT][2];
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) gp[nt][0] = gp[nt][1] = 0.f;
#define AFF_DN_KB(KB)                                                                                  \
  {                                                                                                   \
    uint32_t a[4];                                                                                    \
    aff_frag<B, KB>(w, a);                                                                            \
    _Pragma("unroll") for (int nt = 0; nt < NT; ++nt) {                                                \
      const uint2 bh = ho[nt] >= 0 ? ld8(hb + ho[nt] + 64 * kt + 16 * KB + 4 * c) : make_uint2(0u, 0u); \
      float t[4];                                                                                     \
      mma_z(t, a, bh.x, bh.y);                                                                        \
      const float hs = so[nt] >= 0 ? p.hscale[so[nt] + 4 * kt + KB] : 0.f;                            \
      gp[nt][0] = fmaf(t[0] + t[1], hs, gp[nt][0]);                                                   \
      gp[nt][1] = fmaf(t[2] + t[3], hs, gp[nt][1]);                                                   \
    }                                                                                                 \
  }
    AFF_DN_KB(0)
    AFF_DN_KB(1)
    AFF_DN_KB(2)
    AFF_DN_KB(3)
#undef AFF_DN_KB
    const float s0 = bf16_lo(sb.x) * 0x1p24f, s1 = bf16_hi(sb.x) * 0x1p24f;
    const float b0 = bf16_lo(sb.y), b1 = bf16_hi(sb.y);
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) {
      float hsum = 0.f;
      if (so[nt] >= 0) {
        const float* g = p.hbsum + so[nt] + 4 * kt;
        hsum = ((g[0] + g[1]) + g[2]) + g[3];
      }
      acc[nt][0] = fmaf(s0, gp[nt][0], fmaf(b0, hsum, acc[nt][0]));
      acc[nt][1] = fmaf(s1, gp[nt][1], fmaf(b1, hsum, acc[nt][1]));
    }
  }
#pragma unroll
  for (int nt = 0; nt < NT; ++nt) {
    const int rc = 4 * nt + c;
    if (rc < it.n) {
      float* dst = p.part + (size_t)(it.q0 + rc) * p.d + 16 * it.tile;
      dst[gq] = acc[nt][0];
      dst[gq + 8] = acc[nt][1];
    }
  }
}

template <int B>
__global__ void __launch_bounds__(kAThreads, 2) aff_down_kernel(FwdParams p) {
  pdl_enter();
  extern __shared__ __align__(128) uint8_t sm[];
  const int w = threadIdx.x >> 5;
  AStream ws;
  ws.gw = blockIdx.x * kAW + w;
  ws.nw = gridDim.x * kAW;
  const int total = p.dn_prefix[*p.n_slots];
  ws.n_items = total > ws.gw ? (total - ws.gw + ws.nw - 1) / ws.nw : 0;
  if (ws.n_items == 0) return;
  ws.i = 0;
  aff_seek<B>(p, ws, true);
  uint8_t* ring = sm + (size_t)w * kARingBytes;
  for (int s = 0; s < Aff<B>::kRing; ++s) aff_issue<B>(p, ws, ring + s * Aff<B>::kSlot, true);
  int slot = 0;
  for (int i = 0; i < ws.n_items; ++i) {
    const AItem it = aff_item(p, p.dn_prefix, ws.gw + i * ws.nw, true);
    const int nt = (it.n + 3) / 4;  // 4 block rows (both planes) per n8 tile
    if (nt <= 1) aff_dn_item<B, 1>(p, it, ring, slot, ws);
    else if (nt <= 2) aff_dn_item<B, 2>(p, it, ring, slot, ws);
    else if (nt <= 4) aff_dn_item<B, 4>(p, it, ring, slot, ws);
    else aff_dn_item<B, 8>(p, it, ring, slot, ws);
  }
  cp_wait_all();
}

// ---------------------------------------------------------------- repack

// Code c of a canonical row (little-endian bit stream of b-bit fields).
__device__ __forceinline__ uint32_t canon_code(const uint8_t* row, int b, int c) {
  const long bit = (long)c * b;
  const uint8_t* pb = row + (bit >> 3);
  const int s = (int)(bit & 7);
  uint32_t v = pb[0];
  if (s + b > 8) v |= (uint32_t)pb[1] << 8;
  return (v >> s) & ((1u << b) - 1u);
}

__device__ __forceinline__ bool bf16_finite(uint32_t v) { return (v & 0x7F80u) != 0x7F80u; }

// One thread per (expert, tile, lane): the lane's code words, and (lanes with
// c == 0) its row pair's scale/bias word.
__global__ void repack_affine_kernel(const uint8_t* canon, int n_exp, int d, int f, int b, size_t canon_stride,
                                     uint8_t* out, size_t out_stride, int* err_flag) {
  const int tb = aff_tile_bytes(b);
  const int K64d = d / 64, K64f = f / 64;
  const long n_gu = (long)(f / 16) * K64d * 2, n_dn = (long)(d / 16) * K64f;
  const long per_exp = (n_gu + n_dn) * 32;
  const size_t gu_row = (size_t)d * b / 8, dn_row = (size_t)f * b / 8;
  for (long i = (long)blockIdx.x * blockDim.x + threadIdx.x; i < per_exp * n_exp; i += (long)gridDim.x * blockDim.x) {
    const int e = (int)(i / per_exp);
    const long r = i - (long)e * per_exp;
    const long t = r >> 5;
    const int lane = (int)(r & 31), gq = lane >> 2, c = lane & 3;
    const uint8_t* ce = canon + (size_t)e * canon_stride;
    const uint8_t* dn_codes = ce + (size_t)2 * f * gu_row;
    const uint16_t* gu_sc = reinterpret_cast<const uint16_t*>(dn_codes + (size_t)d * dn_row);
    const uint16_t* dn_sc = gu_sc + (size_t)2 * f * K64d;
    const uint16_t* gu_bi = dn_sc + (size_t)d * K64f;
    const uint16_t* dn_bi = gu_bi + (size_t)2 * f * K64d;
    int row0, kt, ng;
    const uint8_t* codes;
    size_t crow;
    const uint16_t *sc, *bi;
    if (t < n_gu) {
      const int tau = (int)(t / (2 * K64d)), rr = (int)(t % (2 * K64d));
      kt = rr >> 1;
      row0 = (rr & 1) * f + 16 * tau;
      codes = ce;
      crow = gu_row;
      sc = gu_sc;
      bi = gu_bi;
      ng = K64d;
    } else {
      const long t2 = t - n_gu;
      row0 = 16 * (int)(t2 / K64f);
      kt = (int)(t2 % K64f);
      codes = dn_codes;
      crow = dn_row;
      sc = dn_sc;
      bi = dn_bi;
      ng = K64f;
    }
    uint32_t wd[8] = {0u, 0u, 0u, 0u, 0u, 0u, 0u, 0u};
    for (int pi = 0; pi < 16; ++pi) {
      const int kb = pi >> 2, rg = pi & 3;
      const int row = row0 + gq + 8 * (rg & 1);
      const int col = 64 * kt + 16 * kb + 4 * c + 2 * (rg >> 1);
      const uint32_t q0 = canon_code(codes + (size_t)row * crow, b, col);
      const uint32_t q1 = canon_code(codes + (size_t)row * crow, b, col + 1);
      for (int bit = 0; bit < b; ++bit) {
        const int k = b * pi + bit;
        wd[k >> 4] |= ((q0 >> bit) & 1u) << (k & 15);
        wd[k >> 4] |= ((q1 >> bit) & 1u) << (16 + (k & 15));
      }
    }
    uint8_t* dst = out + (size_t)e * out_stride + (size_t)t * tb;
    for (int j = 0; j < b; ++j) reinterpret_cast<uint32_t*>(dst + 4 * (b * lane + j))[0] = wd[j];
    if (c == 0) {
      const size_t g0 = (size_t)(row0 + gq) * ng + kt, g1 = (size_t)(row0 + gq + 8) * ng + kt;
      const uint32_t s0 = sc[g0], s1 = sc[g1], b0 = bi[g0], b1 = bi[g1];
      if (!bf16_finite(s0) || !bf16_finite(s1) || !bf16_finite(b0) || !bf16_finite(b1)) atomicExch(err_flag, 1);
      *reinterpret_cast<uint2*>(dst + 128 * b + 8 * gq) = make_uint2(s0 | (s1 << 16), b0 | (b1 << 16));
    }
  }
}

template <int B>
cudaError_t launch_gu(const FwdParams& p, cudaStream_t stream, int num_sms) {
  aff_gateup_kernel<B><<<2 * num_sms, kAThreads, kASmem, stream>>>(p);
  return cudaGetLastError();
}
template <int B>
cudaError_t launch_dn(const FwdParams& p, cudaStream_t stream, int num_sms) {
  aff_down_kernel<B><<<2 * num_sms, kAThreads, kASmem, stream>>>(p);
  return cudaGetLastError();
}
template <int B>
cudaError_t configure_bits() {
  cudaError_t e = cudaFuncSetAttribute(aff_gateup_kernel<B>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kASmem);
  if (e == cudaSuccess)
    e = cudaFuncSetAttribute(aff_down_kernel<B>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kASmem);
  return e;
}

}  // namespace

// Code widths with compiled kernels.
bool affine_bits_supported(int bits) { return bits == 2 || bits == 3 || bits == 4 || bits == 8; }

cudaError_t configure_affine() {
  cudaError_t e = configure_bits<2>();
  if (e == cudaSuccess) e = configure_bits<3>();
  if (e == cudaSuccess) e = configure_bits<4>();
  if (e == cudaSuccess) e = configure_bits<8>();
  return e;
}

cudaError_t launch_affine_gateup(const FwdParams& p, cudaStream_t stream, int num_sms) {
  switch (p.aff_bits) {
    case 2: return launch_gu<2>(p, stream, num_sms);
    case 3: return launch_gu<3>(p, stream, num_sms);
    case 4: return launch_gu<4>(p, stream, num_sms);
    case 8: return launch_gu<8>(p, stream, num_sms);
    default: return cudaErrorInvalidValue;
  }
}

cudaError_t launch_affine_down(const FwdParams& p, cudaStream_t stream, int num_sms) {
  switch (p.aff_bits) {
    case 2: return launch_dn<2>(p, stream, num_sms);
    case 3: return launch_dn<3>(p, stream, num_sms);
    case 4: return launch_dn<4>(p, stream, num_sms);
    case 8: return launch_dn<8>(p, stream, num_sms);
    default: return cudaErrorInvalidValue;
  }
}

cudaError_t launch_repack_affine(const uint8_t* canon, int n_exp, int d, int f, int bits, size_t canon_stride,
                                 uint8_t* out, size_t out_stride, int* err_flag, cudaStream_t stream) {
  repack_affine_kernel<<<1024, 256, 0, stream>>>(canon, n_exp, d, f, bits, canon_stride, out, out_stride, err_flag);
  return cudaGetLastError();
}

}  // namespace moe
