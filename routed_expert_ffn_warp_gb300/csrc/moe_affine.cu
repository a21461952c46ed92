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
// columns (four k16 MMAs); with the activation group sums stored times 2^-24
// the warp adds s * that + b * (2^-24 sum_c x_c) to its running fp32 sum, and
// the unit's epilogue multiplies the total by 2^24 (exact). The activations are the f16 planes the
// register-decode path already uses: x * 2^sigma_t (one f16 per element) for
// gate/up, and h as two f16 planes with a scale 2^-sh per 16 elements for
// down; the group sums of both come with them.
//
// Work: one CTA per SM takes units in turn (unit u to CTA u % grid), its two
// teams of 8 warps alternate units. Gate/up unit = (slot, one 16-row pair
// tile, block of up to kAffRows rows of the slot): its K range is split over
// the team's 8 warps. Down
// unit = (slot, kADnTiles row tiles, block of rows): warp w takes row tile
// w % kADnTiles and half w / kADnTiles of K. Each warp streams the tiles of
// its share of every unit, in unit order, through its own cp.async ring in
// shared memory, running ahead across units. The warps' partial sums meet in
// shared memory behind one barrier per unit and are added in warp order, so
// every output is a fixed-order sum: results do not depend on the batch or on
// timing. When all of a call's activations fit (decode-sized T), they are
// staged in shared memory once per launch; otherwise the fragments are read
// through L1.
#include <stdint.h>

#include "../../include/moe.h"
#include "moe_device.cuh"
#include "moe_internal.h"

namespace moe {
namespace {

using namespace dev;

constexpr int kAW = 8;                   // warps per team; a team works on one unit at a time
constexpr int kATeams = 2;               // teams per CTA, on alternate units
constexpr int kATeamThreads = kAW * 32;
constexpr int kAThreads = kATeams * kATeamThreads;
constexpr int kARingBytes = 6 * 1024;    // per-warp weight ring
constexpr int kAStageMax = 64 * 1024;    // activations staged in shared memory when they fit in this
constexpr int kADnTiles = kAffDnTiles;   // down: row tiles per unit (each split into kAW / kADnTiles K parts)
constexpr int kAGuNT = kAffRows / 8;     // n8 tiles of a gate/up unit's rows
constexpr int kADnNT = kAffRows / 4;     // n8 tiles of a down unit's rows (both h planes of 4 rows per tile)
constexpr int kAXPad = 16;               // f16 past each staged row: rows 32 bytes past a multiple of 128
constexpr size_t kARings = (size_t)kATeams * kAW * kARingBytes;
constexpr size_t kAGuRedBuf = (size_t)kAW * 2 * kAGuNT * 4 * 32;  // floats of one partial-sum buffer
constexpr size_t kADnRedBuf = (size_t)kAW * kADnNT * 2 * 32;
constexpr size_t kAGuSmemMax = kARings + (size_t)kATeams * 2 * kAGuRedBuf * 4 + kAStageMax + 64;
constexpr size_t kADnSmemMax = kARings + (size_t)kATeams * 2 * kADnRedBuf * 4 + kAStageMax + 64;

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
// Activations: global memory (read-only path) or staged in shared memory (32-bit addresses).
__device__ __forceinline__ uint2 ldg8(const uint16_t* p) { return __ldg(reinterpret_cast<const uint2*>(p)); }
__device__ __forceinline__ uint2 lds8(uint32_t a) {
  uint2 v;
  asm volatile("ld.shared.v2.u32 {%0, %1}, [%2];" : "=r"(v.x), "=r"(v.y) : "r"(a));
  return v;
}
__device__ __forceinline__ float lds4f(uint32_t a) {
  float v;
  asm volatile("ld.shared.f32 %0, [%1];" : "=f"(v) : "r"(a));
  return v;
}
__device__ __forceinline__ float4 lds16f(uint32_t a) {
  float4 v;
  asm volatile("ld.shared.v4.f32 {%0, %1, %2, %3}, [%4];" : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w) : "r"(a));
  return v;
}

__device__ __forceinline__ int token_of_row(const FwdParams& p, int q) { return q < p.P ? p.perm[q] / p.k : q - p.P; }

struct AUnit {
  int e, f;   // expert (E = shared) and its ffn
  int q0, n;  // first h/part row of the block and its rows (<= kAffRows)
  int t0;     // first tile: the pair tile (gate/up) or the first of kADnTiles row tiles (down)
};

__device__ __forceinline__ AUnit aff_unit(const FwdParams& p, const int32_t* prefix, int u, bool down) {
  const int s = find_unit_slot(prefix, *p.n_slots, u);
  const int r = u - prefix[s];
  AUnit un;
  un.e = p.slot_expert[s];
  un.f = un.e == p.E ? p.S : p.F;
  const int groups = down ? (p.d / 16 + kADnTiles - 1) / kADnTiles : un.f / 16;
  const int blk = r / groups;
  un.t0 = (r - blk * groups) * (down ? kADnTiles : 1);
  un.q0 = p.slot_q0[s] + kAffRows * blk;
  un.n = min(kAffRows, p.slot_n[s] - kAffRows * blk);
  return un;
}

__device__ __forceinline__ void k_range(int K64, int part, int parts, int& k0, int& k1) {
  k0 = K64 * part / parts;
  k1 = K64 * (part + 1) / parts;
}

// Where warp w's share of a unit lies: gate/up -- k tiles [k0, k1) of the pair
// tile; down -- row tile m, k tiles [k0, k1).
struct Share {
  int m, k0, k1;
};
__device__ __forceinline__ Share gu_share(const FwdParams& p, const AUnit& un, int w) {
  Share sh;
  sh.m = un.t0;
  k_range(p.d / 64, w, kAW, sh.k0, sh.k1);
  return sh;
}
__device__ __forceinline__ Share dn_share(const FwdParams& p, const AUnit& un, int w) {
  Share sh;
  sh.m = un.t0 + w % kADnTiles;
  k_range(un.f / 64, w / kADnTiles, kAW / kADnTiles, sh.k0, sh.k1);
  if (sh.m >= p.d / 16) sh.k1 = sh.k0;
  return sh;
}

// The weight stream of one warp: its shares of the CTA's units in order, two
// tiles per ring slot (gate/up: the gate and up tiles of one k tile; down: two
// k tiles of the row tile, one at the end of an odd count).
struct AStream {
  int i, n_units;  // CTA-local index of the unit being issued (the team's: every kATeams-th), unit count
  const uint8_t* src;
  int left;        // tiles of that share still to issue
};

template <int B, bool DOWN>
__device__ __forceinline__ void aff_seek(const FwdParams& p, AStream& ws) {
  const int w = (threadIdx.x >> 5) % kAW;
  for (; ws.i < ws.n_units; ws.i += kATeams) {
    const AUnit un = aff_unit(p, DOWN ? p.dn_prefix : p.gu_prefix, blockIdx.x + ws.i * gridDim.x, DOWN);
    const Share sh = DOWN ? dn_share(p, un, w) : gu_share(p, un, w);
    if (sh.k1 <= sh.k0) continue;
    const uint8_t* base = p.packed + (size_t)weight_index(p, un.e) * p.expert_stride;
    if (DOWN) {
      ws.src = base + aff_gu_bytes(p.d, un.f, B) + ((size_t)sh.m * (un.f / 64) + sh.k0) * Aff<B>::kTile;
      ws.left = sh.k1 - sh.k0;
    } else {
      ws.src = base + ((size_t)sh.m * (p.d / 64) + sh.k0) * Aff<B>::kSlot;
      ws.left = 2 * (sh.k1 - sh.k0);
    }
    return;
  }
}

template <int B, bool DOWN>
__device__ __forceinline__ void aff_issue(const FwdParams& p, AStream& ws, uint8_t* dst) {
  const int lane = threadIdx.x & 31;
  if (ws.i < ws.n_units) {
    const int nt = min(2, ws.left), n16 = nt * Aff<B>::kTile / 16;
#pragma unroll
    for (int r = 0; r < (Aff<B>::kSlot / 16 + 31) / 32; ++r)
      if (lane + 32 * r < n16) cp16(dst + 16 * (lane + 32 * r), ws.src + 16 * (lane + 32 * r));
    ws.src += nt * Aff<B>::kTile;
    ws.left -= nt;
    if (ws.left == 0) {
      ws.i += kATeams;
      aff_seek<B, DOWN>(p, ws);
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

// Activations of the launch: in shared memory when staged, else in global memory.
// Staged, every array is followed by one row of zeros (row T, 2Q or Q) that
// absent rows read; from global memory they read p.zeros.
struct Act {
  const uint16_t* x;   // gate/up: x16 rows of tokens, xrow f16 apart
  int xrow;
  const float* xg;     // their group sums, xgrow floats apart
  int xgrow;
  const uint16_t* h;   // down: h rows (2 q + plane), hrow f16 apart
  int hrow;
  const float* hs;     // h scales and group sums per row q, hgrow floats apart
  const float* hb;
  int hgrow;
  const uint16_t* zx;  // the zero rows of x (h) and of the per-row floats
  const float* zf;
};

// Copy `rows` rows of `bytes` bytes (both strides multiples of 16) with all threads.
__device__ __forceinline__ void stage_rows(void* dst, int dst_stride, const void* src, int src_stride, int rows,
                                           int bytes) {
  const int per = bytes / 16;
  for (int i = threadIdx.x; i < rows * per; i += kAThreads) {
    const int r = i / per, c = i - r * per;
    cp16(static_cast<uint8_t*>(dst) + (size_t)r * dst_stride + 16 * c,
         static_cast<const uint8_t*>(src) + (size_t)r * src_stride + 16 * c);
  }
}

// Bytes of the staged activations of a call (0: they are read from global memory).
__host__ __device__ inline int gu_stage_bytes(const FwdParams& p) {
  const size_t b = (size_t)(p.T + 1) * (p.d64 + kAXPad) * 2 + (size_t)(p.T + 1) * p.xg_pitch * 4;
  return b <= (size_t)kAStageMax ? (int)b : 0;
}
__host__ __device__ inline int dn_rows(const FwdParams& p) { return p.P + ((p.S > 0 && p.e_begin == 0) ? p.T : 0); }
__host__ __device__ inline int dn_stage_bytes(const FwdParams& p) {
  const size_t q = (size_t)dn_rows(p);
  const size_t b = (2 * q + 1) * (p.fmax64 + kAXPad) * 2 + (q + 1) * p.hgroups * 4 * 2;
  return b <= (size_t)kAStageMax ? (int)b : 0;
}

// ---------------------------------------------------------------- gate/up

template <int B, int NT, bool S>
__device__ void gu_share_compute(const FwdParams& p, const AUnit& un, const Share& sh, uint8_t* ring, int& slot,
                                 AStream& ws, const Act& A, float* red) {
  const int lane = threadIdx.x & 31, w = (threadIdx.x >> 5) % kAW, gq = lane >> 2, c = lane & 3;
  const uint16_t* xr[NT];  // B fragment row 8 nt + gq: its token's x row (a zero row past the block)
  const float* xs[NT][2];  // C fragment column 8 nt + 2c + j: its token's group sums (zeros past the block)
  uint32_t xa[NT], sa[NT][2];  // the same as shared-memory addresses (staged)
#pragma unroll
  for (int nt = 0; nt < NT; ++nt) {
    const int m = 8 * nt + gq;
    xr[nt] = (m < un.n ? A.x + (size_t)token_of_row(p, un.q0 + m) * A.xrow : A.zx) + 4 * c;
#pragma unroll
    for (int j = 0; j < 2; ++j) {
      const int mc = 8 * nt + 2 * c + j;
      xs[nt][j] = mc < un.n ? A.xg + (size_t)token_of_row(p, un.q0 + mc) * A.xgrow : A.zf;
      if (S) sa[nt][j] = smem_u32(xs[nt][j]);
    }
    if (S) xa[nt] = smem_u32(xr[nt]);
  }
  float acc[2][NT][4];
#pragma unroll
  for (int h = 0; h < 2; ++h)
#pragma unroll
    for (int nt = 0; nt < NT; ++nt)
#pragma unroll
      for (int r = 0; r < 4; ++r) acc[h][nt][r] = 0.f;
  for (int kt = sh.k0; kt < sh.k1; ++kt) {
    cp_wait<Aff<B>::kRing - 1>();
    __syncwarp();
    uint32_t wd[2][B];
    uint2 sb[2];
    const uint8_t* sl = ring + slot * Aff<B>::kSlot;
    load_tile<B>(sl, lane, wd[0], sb[0]);
    load_tile<B>(sl + Aff<B>::kTile, lane, wd[1], sb[1]);
    __syncwarp();
    aff_issue<B, false>(p, ws, ring + slot * Aff<B>::kSlot);
    if (++slot == Aff<B>::kRing) slot = 0;
    // two accumulators per (matrix, n8 tile): k16 blocks 0 + 2 and 1 + 3
    float t[2][2][NT][4];
#define AFF_GU_KB(KB)                                                                                    \
  {                                                                                                     \
    uint32_t a0[4], a1[4];                                                                              \
    aff_frag<B, KB>(wd[0], a0);                                                                         \
    aff_frag<B, KB>(wd[1], a1);                                                                         \
    _Pragma("unroll") for (int nt = 0; nt < NT; ++nt) {                                                  \
      const uint2 bx = S ? lds8(xa[nt] + 2 * (64 * kt + 16 * KB)) : ldg8(xr[nt] + 64 * kt + 16 * KB);    \
      if (KB < 2) {                                                                                     \
        mma_z(t[KB & 1][0][nt], a0, bx.x, bx.y);                                                        \
        mma_z(t[KB & 1][1][nt], a1, bx.x, bx.y);                                                        \
      } else {                                                                                          \
        mma16816(t[KB & 1][0][nt], a0, bx.x, bx.y);                                                     \
        mma16816(t[KB & 1][1][nt], a1, bx.x, bx.y);                                                     \
      }                                                                                                 \
    }                                                                                                   \
  }
    AFF_GU_KB(0)
    AFF_GU_KB(1)
    AFF_GU_KB(2)
    AFF_GU_KB(3)
#undef AFF_GU_KB
    // the group's affine terms: rows gq (C registers 0, 1) and gq + 8 (2, 3)
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) {
      const float xs0 = S ? lds4f(sa[nt][0] + 4 * kt) : __ldg(xs[nt][0] + kt);
      const float xs1 = S ? lds4f(sa[nt][1] + 4 * kt) : __ldg(xs[nt][1] + kt);
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        const float s0 = bf16_lo(sb[h].x), s1 = bf16_hi(sb[h].x);
        const float b0 = bf16_lo(sb[h].y), b1 = bf16_hi(sb[h].y);
        acc[h][nt][0] = fmaf(s0, t[0][h][nt][0] + t[1][h][nt][0], fmaf(b0, xs0, acc[h][nt][0]));
        acc[h][nt][1] = fmaf(s0, t[0][h][nt][1] + t[1][h][nt][1], fmaf(b0, xs1, acc[h][nt][1]));
        acc[h][nt][2] = fmaf(s1, t[0][h][nt][2] + t[1][h][nt][2], fmaf(b1, xs0, acc[h][nt][2]));
        acc[h][nt][3] = fmaf(s1, t[0][h][nt][3] + t[1][h][nt][3], fmaf(b1, xs1, acc[h][nt][3]));
      }
    }
  }
  // this warp's partial sums: red[w][h][nt][r][lane]
#pragma unroll
  for (int h = 0; h < 2; ++h)
#pragma unroll
    for (int nt = 0; nt < NT; ++nt)
#pragma unroll
      for (int r = 0; r < 4; ++r) red[(((size_t)w * 2 + h) * kAGuNT + nt) * 4 * 32 + r * 32 + lane] = acc[h][nt][r];
}

// SwiGLU epilogue of a unit (one warp): the warps' partial sums added in warp
// order, then h rows 16 tau + gq (+ 8) of the block's rows 8 nt + 2c (+ 1),
// stored as the down GEMM reads them (two f16 planes, a 2^-sh scale and the
// group sum per 16 elements).
template <int NT>
__device__ void gu_epilogue(const FwdParams& p, const AUnit& un, const float* red) {
  const int lane = threadIdx.x & 31, gq = lane >> 2, c = lane & 3;
  const int tau = un.t0;
#pragma unroll
  for (int nt = 0; nt < NT; ++nt) {
#pragma unroll
    for (int col = 0; col < 2; ++col) {
      const int m = 8 * nt + 2 * c + col;
      const bool ok = m < un.n;
      const float xi = ok ? p.xinv[token_of_row(p, un.q0 + m)] * 0x1p24f : 0.f;
      float hv[2];
#pragma unroll
      for (int r = 0; r < 2; ++r) {
        float g = 0.f, u = 0.f;
#pragma unroll
        for (int w = 0; w < kAW; ++w) {
          g += red[(((size_t)w * 2 + 0) * kAGuNT + nt) * 4 * 32 + (2 * r + col) * 32 + lane];
          u += red[(((size_t)w * 2 + 1) * kAGuNT + nt) * 4 * 32 + (2 * r + col) * 32 + lane];
        }
        const float gate = g * xi, up = u * xi;  // xi carries the 2^24 of the sums
        hv[r] = ok ? gate / (1.f + expf(-gate)) * up : 0.f;
      }
      float mx = fmaxf(fabsf(hv[0]), fabsf(hv[1]));
#pragma unroll
      for (int o = 4; o < 32; o <<= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
      const int sh = f16_headroom_exponent(mx);
      const float sc = pow2f(sh);
      __half* hi = reinterpret_cast<__half*>(p.hbuf) + (size_t)(un.q0 + m) * 2 * p.fmax64;
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
        const size_t q = (size_t)(un.q0 + m) * p.hgroups + tau;
        p.hscale[q] = pow2f(-sh);
        p.hbsum[q] = rep * pow2f(-sh) * 0x1p-24f;
      }
    }
  }
}

template <int B>
__global__ void __launch_bounds__(kAThreads, 1) aff_gateup_kernel(FwdParams p) {
  pdl_enter();
  extern __shared__ __align__(128) uint8_t sm[];
  const int gw = threadIdx.x >> 5, w = gw % kAW, team = gw / kAW;
  const int total = p.gu_prefix[*p.n_slots];
  const int n_units = total > (int)blockIdx.x ? (total - (int)blockIdx.x + gridDim.x - 1) / gridDim.x : 0;
  if (n_units == 0) return;
  float* red = reinterpret_cast<float*>(sm + kARings) + (size_t)team * 2 * kAGuRedBuf;
  uint8_t* stage = sm + kARings + (size_t)kATeams * 2 * kAGuRedBuf * 4;
  uint64_t* sbar = reinterpret_cast<uint64_t*>(stage + kAStageMax);
  Act A{};
  const int stage_bytes = gu_stage_bytes(p);
  if (stage_bytes) {  // x16 and its group sums of every token (+ a zero row each), before the weight streams
    A.xrow = p.d64 + kAXPad;
    A.xgrow = p.xg_pitch;
    uint16_t* xs = reinterpret_cast<uint16_t*>(stage);
    float* xg = reinterpret_cast<float*>(stage + (size_t)(p.T + 1) * A.xrow * 2);
    A.x = xs;
    A.xg = xg;
    A.zx = xs + (size_t)p.T * A.xrow;
    A.zf = xg + (size_t)p.T * A.xgrow;
    if (threadIdx.x == 0) {
      mbar_init(sbar, kAThreads);
      fence_mbar_init();
    }
    for (int i = threadIdx.x; i < A.xrow; i += kAThreads) const_cast<uint16_t*>(A.zx)[i] = 0;
    for (int i = threadIdx.x; i < A.xgrow; i += kAThreads) const_cast<float*>(A.zf)[i] = 0.f;
    __syncthreads();
    stage_rows(xs, A.xrow * 2, p.x16, p.d64 * 2, p.T, p.d64 * 2);
    stage_rows(xg, A.xgrow * 4, p.xgsum, p.xg_pitch * 4, p.T, p.xg_pitch * 4);
    cp_arrive(sbar);
  } else {
    A.x = p.x16;
    A.xrow = p.d64;
    A.xg = p.xgsum;
    A.xgrow = p.xg_pitch;
    A.zx = static_cast<const uint16_t*>(p.zeros);
    A.zf = static_cast<const float*>(p.zeros);
  }
  AStream ws;
  ws.i = team;
  ws.n_units = n_units;
  aff_seek<B, false>(p, ws);
  uint8_t* ring = sm + (size_t)gw * kARingBytes;
  for (int s = 0; s < Aff<B>::kRing; ++s) aff_issue<B, false>(p, ws, ring + s * Aff<B>::kSlot);
  if (stage_bytes) wait_chunk(sbar, 0, p.status);
  int slot = 0;
  for (int i = team, j = 0; i < n_units; i += kATeams, ++j) {
    const AUnit un = aff_unit(p, p.gu_prefix, blockIdx.x + i * gridDim.x, false);
    const Share sh = gu_share(p, un, w);
    float* rb = red + (size_t)(j & 1) * kAGuRedBuf;
    if (stage_bytes) {
      if (un.n <= 8) gu_share_compute<B, 1, true>(p, un, sh, ring, slot, ws, A, rb);
      else gu_share_compute<B, 2, true>(p, un, sh, ring, slot, ws, A, rb);
    } else {
      if (un.n <= 8) gu_share_compute<B, 1, false>(p, un, sh, ring, slot, ws, A, rb);
      else gu_share_compute<B, 2, false>(p, un, sh, ring, slot, ws, A, rb);
    }
    named_bar(1 + team, kATeamThreads);  // every warp's partial sums of the unit are in rb
    if (w == j % kAW) {
      if (un.n <= 8) gu_epilogue<1>(p, un, rb);
      else gu_epilogue<2>(p, un, rb);
    }
  }
  cp_wait_all();
}

// ---------------------------------------------------------------- down

template <int B, int NT, bool S>
__device__ void dn_share_compute(const FwdParams& p, const AUnit& un, const Share& sh, uint8_t* ring, int& slot,
                                 AStream& ws, const Act& A, float* red) {
  const int lane = threadIdx.x & 31, w = (threadIdx.x >> 5) % kAW, gq = lane >> 2, c = lane & 3;
  const uint16_t* hr[NT];  // B fragment row gq of n8 tile nt = (block row 4 nt + gq / 2, plane gq % 2)
  const float* hsr[NT];    // C fragment columns 2c, 2c + 1 = both planes of block row 4 nt + c: its scales
  const float* hbr[NT];    // ... and group sums (zero rows past the block)
  uint32_t ha[NT], hsa[NT], hba[NT];  // the same as shared-memory addresses (staged)
#pragma unroll
  for (int nt = 0; nt < NT; ++nt) {
    const int r = 4 * nt + (gq >> 1), rc = 4 * nt + c;
    hr[nt] = (r < un.n ? A.h + (size_t)((un.q0 + r) * 2 + (gq & 1)) * A.hrow : A.zx) + 4 * c;
    hsr[nt] = rc < un.n ? A.hs + (size_t)(un.q0 + rc) * A.hgrow : A.zf;
    hbr[nt] = rc < un.n ? A.hb + (size_t)(un.q0 + rc) * A.hgrow : A.zf;
    if (S) {
      ha[nt] = smem_u32(hr[nt]);
      hsa[nt] = smem_u32(hsr[nt]);
      hba[nt] = smem_u32(hbr[nt]);
    }
  }
  float acc[NT][2];
#pragma unroll
  for (int nt = 0; nt < NT; ++nt) acc[nt][0] = acc[nt][1] = 0.f;
  int in_slot = 0;
  for (int kt = sh.k0; kt < sh.k1; ++kt) {
    if (in_slot == 0) {
      cp_wait<Aff<B>::kRing - 1>();
      __syncwarp();
    }
    uint32_t wd[B];
    uint2 sb;
    load_tile<B>(ring + slot * Aff<B>::kSlot + in_slot * Aff<B>::kTile, lane, wd, sb);
    if (++in_slot == 2 || kt + 1 == sh.k1) {
      in_slot = 0;
      __syncwarp();
      aff_issue<B, true>(p, ws, ring + slot * Aff<B>::kSlot);
      if (++slot == Aff<B>::kRing) slot = 0;
    }
    float gp[NT][2];
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) gp[nt][0] = gp[nt][1] = 0.f;
#define AFF_DN_KB(KB)                                                                                    \
  {                                                                                                     \
    uint32_t a[4];                                                                                      \
    aff_frag<B, KB>(wd, a);                                                                             \
    _Pragma("unroll") for (int nt = 0; nt < NT; ++nt) {                                                  \
      const uint2 bh = S ? lds8(ha[nt] + 2 * (64 * kt + 16 * KB)) : ldg8(hr[nt] + 64 * kt + 16 * KB);    \
      float t[4];                                                                                       \
      mma_z(t, a, bh.x, bh.y);                                                                          \
      const float hs = S ? lds4f(hsa[nt] + 4 * (4 * kt + KB)) : __ldg(hsr[nt] + 4 * kt + KB);            \
      gp[nt][0] = fmaf(t[0] + t[1], hs, gp[nt][0]);                                                     \
      gp[nt][1] = fmaf(t[2] + t[3], hs, gp[nt][1]);                                                     \
    }                                                                                                   \
  }
    AFF_DN_KB(0)
    AFF_DN_KB(1)
    AFF_DN_KB(2)
    AFF_DN_KB(3)
#undef AFF_DN_KB
    const float s0 = bf16_lo(sb.x), s1 = bf16_hi(sb.x);
    const float b0 = bf16_lo(sb.y), b1 = bf16_hi(sb.y);
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) {
      const float4 g = S ? lds16f(hba[nt] + 16 * kt) : __ldg(reinterpret_cast<const float4*>(hbr[nt] + 4 * kt));
      const float hsum = ((g.x + g.y) + g.z) + g.w;
      acc[nt][0] = fmaf(s0, gp[nt][0], fmaf(b0, hsum, acc[nt][0]));
      acc[nt][1] = fmaf(s1, gp[nt][1], fmaf(b1, hsum, acc[nt][1]));
    }
  }
#pragma unroll
  for (int nt = 0; nt < NT; ++nt) {
    red[(((size_t)w * kADnNT + nt) * 2 + 0) * 32 + lane] = acc[nt][0];
    red[(((size_t)w * kADnNT + nt) * 2 + 1) * 32 + lane] = acc[nt][1];
  }
}

// The down unit's outputs (warps 0 .. kADnTiles - 1, one row tile each): the
// K parts added in order, rows 16 m + gq (+ 8) of block rows 4 nt + c.
template <int NT>
__device__ void dn_epilogue(const FwdParams& p, const AUnit& un, const float* red) {
  const int lane = threadIdx.x & 31, w = (threadIdx.x >> 5) % kAW, gq = lane >> 2, c = lane & 3;
  const int m = un.t0 + w;
  if (m >= p.d / 16) return;
#pragma unroll
  for (int nt = 0; nt < NT; ++nt) {
    const int rc = 4 * nt + c;
    float v0 = 0.f, v1 = 0.f;
#pragma unroll
    for (int k = 0; k < kAW / kADnTiles; ++k) {
      const int ww = w + kADnTiles * k;
      v0 += red[(((size_t)ww * kADnNT + nt) * 2 + 0) * 32 + lane];
      v1 += red[(((size_t)ww * kADnNT + nt) * 2 + 1) * 32 + lane];
    }
    if (rc < un.n) {  // the sums carry 2^-24 (codes as f16 subnormals, h group sums scaled to match)
      float* dst = p.part + (size_t)(un.q0 + rc) * p.d + 16 * m;
      dst[gq] = v0 * 0x1p24f;
      dst[gq + 8] = v1 * 0x1p24f;
    }
  }
}

template <int B>
__global__ void __launch_bounds__(kAThreads, 1) aff_down_kernel(FwdParams p) {
  pdl_enter();
  extern __shared__ __align__(128) uint8_t sm[];
  const int gw = threadIdx.x >> 5, w = gw % kAW, team = gw / kAW;
  const int total = p.dn_prefix[*p.n_slots];
  const int n_units = total > (int)blockIdx.x ? (total - (int)blockIdx.x + gridDim.x - 1) / gridDim.x : 0;
  if (n_units == 0) return;
  float* red = reinterpret_cast<float*>(sm + kARings) + (size_t)team * 2 * kADnRedBuf;
  uint8_t* stage = sm + kARings + (size_t)kATeams * 2 * kADnRedBuf * 4;
  uint64_t* sbar = reinterpret_cast<uint64_t*>(stage + kAStageMax);
  Act A{};
  const int stage_bytes = dn_stage_bytes(p);
  if (stage_bytes) {  // both h planes, scales and group sums of every row (+ zero rows), before the weight streams
    const int Q = dn_rows(p);
    A.hrow = p.fmax64 + kAXPad;
    A.hgrow = p.hgroups;
    uint16_t* hs = reinterpret_cast<uint16_t*>(stage);
    float* sc = reinterpret_cast<float*>(stage + (size_t)(2 * Q + 1) * A.hrow * 2);
    float* gs = sc + (size_t)(Q + 1) * A.hgrow;
    A.h = hs;
    A.hs = sc;
    A.hb = gs;
    A.zx = hs + (size_t)2 * Q * A.hrow;
    A.zf = sc + (size_t)Q * A.hgrow;
    if (threadIdx.x == 0) {
      mbar_init(sbar, kAThreads);
      fence_mbar_init();
    }
    for (int i = threadIdx.x; i < A.hrow; i += kAThreads) const_cast<uint16_t*>(A.zx)[i] = 0;
    for (int i = threadIdx.x; i < A.hgrow; i += kAThreads) const_cast<float*>(A.zf)[i] = 0.f;
    __syncthreads();
    stage_rows(hs, A.hrow * 2, p.hbuf, p.fmax64 * 2, 2 * Q, p.fmax64 * 2);
    stage_rows(sc, A.hgrow * 4, p.hscale, p.hgroups * 4, Q, p.hgroups * 4);
    stage_rows(gs, A.hgrow * 4, p.hbsum, p.hgroups * 4, Q, p.hgroups * 4);
    cp_arrive(sbar);
  } else {
    A.h = p.hbuf;
    A.hrow = p.fmax64;
    A.hs = p.hscale;
    A.hb = p.hbsum;
    A.hgrow = p.hgroups;
    A.zx = static_cast<const uint16_t*>(p.zeros);
    A.zf = static_cast<const float*>(p.zeros);
  }
  AStream ws;
  ws.i = team;
  ws.n_units = n_units;
  aff_seek<B, true>(p, ws);
  uint8_t* ring = sm + (size_t)gw * kARingBytes;
  for (int s = 0; s < Aff<B>::kRing; ++s) aff_issue<B, true>(p, ws, ring + s * Aff<B>::kSlot);
  if (stage_bytes) wait_chunk(sbar, 0, p.status);
  int slot = 0;
  for (int i = team, j = 0; i < n_units; i += kATeams, ++j) {
    const AUnit un = aff_unit(p, p.dn_prefix, blockIdx.x + i * gridDim.x, true);
    const Share sh = dn_share(p, un, w);
    float* rb = red + (size_t)(j & 1) * kADnRedBuf;
    const int nt = (un.n + 3) / 4;  // 4 block rows (both planes) per n8 tile
    if (stage_bytes) {
      if (nt <= 1) dn_share_compute<B, 1, true>(p, un, sh, ring, slot, ws, A, rb);
      else if (nt <= 2) dn_share_compute<B, 2, true>(p, un, sh, ring, slot, ws, A, rb);
      else dn_share_compute<B, 4, true>(p, un, sh, ring, slot, ws, A, rb);
    } else {
      if (nt <= 1) dn_share_compute<B, 1, false>(p, un, sh, ring, slot, ws, A, rb);
      else if (nt <= 2) dn_share_compute<B, 2, false>(p, un, sh, ring, slot, ws, A, rb);
      else dn_share_compute<B, 4, false>(p, un, sh, ring, slot, ws, A, rb);
    }
    named_bar(1 + team, kATeamThreads);  // every warp's partial sums of the unit are in rb
    if (w < kADnTiles) {
      if (nt <= 1) dn_epilogue<1>(p, un, rb);
      else if (nt <= 2) dn_epilogue<2>(p, un, rb);
      else dn_epilogue<4>(p, un, rb);
    }
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

// Both GEMMs join the forward chain's programmatic launches: each may be
// scheduled while the grid before it drains and waits for it (pdl_enter)
// before reading anything that grid wrote.
template <int B>
cudaError_t launch_gu(const FwdParams& p, cudaStream_t stream, int num_sms) {
  return launch_chained(aff_gateup_kernel<B>, dim3(num_sms), dim3(kAThreads), kAGuSmemMax, stream, p);
}
template <int B>
cudaError_t launch_dn(const FwdParams& p, cudaStream_t stream, int num_sms) {
  return launch_chained(aff_down_kernel<B>, dim3(num_sms), dim3(kAThreads), kADnSmemMax, stream, p);
}
template <int B>
cudaError_t configure_bits() {
  cudaError_t e =
      cudaFuncSetAttribute(aff_gateup_kernel<B>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kAGuSmemMax);
  if (e == cudaSuccess)
    e = cudaFuncSetAttribute(aff_down_kernel<B>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kADnSmemMax);
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
