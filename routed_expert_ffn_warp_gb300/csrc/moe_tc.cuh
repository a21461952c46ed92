// tcgen05 (5th-generation tensor core) helpers: TMEM allocation, shared
// memory matrix descriptors, block-scaled MMA of MXFP4 weights by MXFP8
// activations, commit to an mbarrier, TMEM loads and stores, fences.
//
// Conventions used by every caller (K-major operands, no swizzle):
//  * an operand tile is an array of core matrices of 8 rows x 16 bytes (128
//    contiguous bytes); for MXFP4 a 16-byte row holds 16 E2M1 codes packed in
//    its first 8 bytes (low nibble = even element) and 8 bytes of padding; for
//    MXFP8 it holds 16 E4M3 bytes;
//  * core matrices adjacent along K are LBO bytes apart, 8-row groups SBO
//    bytes apart;
//  * scale factors (one E8M0 byte per row and 32-element K block) live in
//    TMEM: for rows 32 r + l, byte b of column base + r in lane l holds the
//    scale of K block b, replicated in all four lane quadrants (four warps,
//    one per quadrant, each storing 512-byte blocks [lane][4 words] with
//    tcgen05.st); the MMA picks the byte with the scale-factor ids of its
//    instruction descriptor.
#pragma once
#include <stdint.h>

#include "../../include/moe.h"
#include "moe_device.cuh"

namespace moe {
namespace tc {

using dev::smem_u32;

__device__ __forceinline__ uint64_t smem_desc(const void* p, uint32_t lbo, uint32_t sbo) {
  return (uint64_t)((smem_u32(p) & 0x3FFFFu) >> 4) | ((uint64_t)(lbo >> 4) << 16) | ((uint64_t)(sbo >> 4) << 32) |
         (1ull << 46);
}

// Instruction descriptor of kind::mxf8f6f4 with A = E2M1, B = E4M3, UE8M0
// scales, K-major A and B, M x N, scale-factor ids a_id / b_id.
__device__ __forceinline__ uint32_t idesc_mxf4_mxf8(int M, int N, int a_id, int b_id) {
  return (5u << 7) | (0u << 10) | ((uint32_t)(N >> 3) << 17) | (1u << 23) | ((uint32_t)(M >> 4) << 24) |
         ((uint32_t)b_id << 4) | ((uint32_t)a_id << 29);
}

__device__ __forceinline__ void alloc(uint32_t* slot, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(slot)), "r"(ncols)
               : "memory");
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void dealloc(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols) : "memory");
}
__device__ __forceinline__ void fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }
// generic-proxy writes to shared memory (cp.async, st.shared) -> visible to the tensor core
__device__ __forceinline__ void fence_proxy_async() { asm volatile("fence.proxy.async.shared::cta;" ::: "memory"); }

__device__ __forceinline__ void mma_mxf4_mxf8(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc, uint32_t idesc,
                                              uint32_t sfa_tmem, uint32_t sfb_tmem, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %6, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::mxf8f6f4.block_scale.scale_vec::1X [%0], %1, %2, %3, [%4], [%5], p;\n\t}" ::"r"(
          d_tmem),
      "l"(adesc), "l"(bdesc), "r"(idesc), "r"(sfa_tmem), "r"(sfb_tmem), "r"(accumulate)
      : "memory");
}
// Copy a 512-byte block of shared memory, 32 rows of 16 bytes (8-row groups
// 128 bytes apart: the descriptor smem_desc(block, 128, 128)), to TMEM lanes
// 0..31 of 4 consecutive columns at taddr, replicated into all four lane
// quadrants: the scale-factor layout of the block-scaled MMAs. It runs in
// issue order with the MMAs the same thread issues after it; taddr's column
// must be a multiple of 4.
__device__ __forceinline__ void cp_32x128b_x4(uint32_t taddr, uint64_t sdesc) {
  asm volatile("tcgen05.cp.cta_group::1.32x128b.warpx4 [%0], %1;" ::"r"(taddr), "l"(sdesc) : "memory");
}
// TMA tiled load of the box at (x, y) of a 2-D tensor map (a kernel parameter
// declared __grid_constant__) into this CTA's shared memory; completion is
// signalled on `bar` as transaction bytes.
__device__ __forceinline__ void tma_load_2d(void* dst, const void* map, int x, int y, uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], [%4];" ::"r"(
          smem_u32(dst)),
      "l"(map), "r"(x), "r"(y), "r"(smem_u32(bar))
      : "memory");
}
// The same for the box at (x, y, z) of a 3-D tensor map.
__device__ __forceinline__ void tma_load_3d(void* dst, const void* map, int x, int y, int z, uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3, %4}], "
      "[%5];" ::"r"(smem_u32(dst)),
      "l"(map), "r"(x), "r"(y), "r"(z), "r"(smem_u32(bar))
      : "memory");
}
// Arrive once on `bar` when every tcgen05 operation issued so far by this thread has completed.
__device__ __forceinline__ void commit(uint64_t* bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(smem_u32(bar))
               : "memory");
}

__device__ __forceinline__ void st4(uint32_t taddr, uint32_t a, uint32_t b, uint32_t c, uint32_t d) {
  asm volatile("tcgen05.st.sync.aligned.32x32b.x4.b32 [%0], {%1, %2, %3, %4};" ::"r"(taddr), "r"(a), "r"(b), "r"(c),
               "r"(d)
               : "memory");
}
__device__ __forceinline__ void wait_st() { asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory"); }

// 16 consecutive 32-bit columns of this warp's 32 lanes.
__device__ __forceinline__ void ld16(uint32_t taddr, float (&v)[16]) {
  uint32_t r[16];
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]), "=r"(r[8]),
        "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
      : "r"(taddr));
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
  for (int i = 0; i < 16; ++i) v[i] = __uint_as_float(r[i]);
}

// ---------------------------------------------------------------- bounded mbarrier waits

using dev::globaltimer;
using dev::mbar_try_wait;
using dev::mbar_try_wait_hint;
constexpr long long kTcWaitNs = 50000000LL;  // 50 ms: orders of magnitude above any wait of a healthy layer

// Bounded mbarrier waits. Every role passes every phase of the barriers it
// waits on in order, so a parity wait never meets a phase two steps old. On
// expiry the wait records MOE_ERR_TIMEOUT, raises the CTA's abort flag and
// returns false; once the flag is up every wait returns false at once and
// every role stops issuing copies and MMAs (the kernel then drains what is in
// flight before it frees tensor memory, see the end of gemm_tc_kernel).
__device__ __forceinline__ bool bounded_wait(uint64_t* bar, uint32_t parity, int* status, volatile int* abort) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = globaltimer();
  while (!mbar_try_wait(bar, parity)) {
    if (*abort) return false;
    if ((long long)(globaltimer() - t0) > kTcWaitNs) {
      *abort = 1;
      atomicCAS(status, 0, MOE_ERR_TIMEOUT);
      return false;
    }
  }
  return true;
}
// The same wait for the roles off the MMA lanes' critical path (producers,
// epilogue): each try may suspend the thread for up to 20 us until the phase
// completes, so that waiting warps leave their issue slots to the MMA lanes.
__device__ __forceinline__ bool bounded_wait_sleep(uint64_t* bar, uint32_t parity, int* status, volatile int* abort) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = globaltimer();
  while (!mbar_try_wait_hint(bar, parity, 20000u)) {
    if (*abort) return false;
    if ((long long)(globaltimer() - t0) > kTcWaitNs) {
      *abort = 1;
      atomicCAS(status, 0, MOE_ERR_TIMEOUT);
      return false;
    }
  }
  return true;
}
// After an abort: long enough for every copy and MMA already issued to land
// (each takes microseconds), so that no copy writes into shared memory and no
// MMA touches tensor memory after this CTA has freed them.
constexpr long long kDrainNs = 1000000LL;

// ---------------------------------------------------------------- MXFP8 planes of a 32-element block

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


// Split the 32 values of a block (one per lane) into 4 MXFP8 planes with one
// reduction: plane 0 takes the block maximum into [128, 256) as above; every
// later plane's scale is the previous one divided by 32. An E4M3 code of a
// value below 256 errs by at most 8 (half its spacing there), so a plane's
// remainder, scaled by 32, stays at most 256 and fits the next plane; after
// the 4 planes the error is below 2^-19 of the block maximum.
__device__ __forceinline__ void split_planes4_fixed(float v, uint32_t (&code)[4], uint32_t (&sc)[4]) {
  float amax = fabsf(v);
  for (int o = 16; o; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
  int sh = amax > 0.f ? (int)((__float_as_uint(amax) >> 23) & 0xFF) - 127 - 7 : 0;
#pragma unroll
  for (int pl = 0; pl < 4; ++pl) {
    const int s = max(-127, min(127, sh));
    const float ish = __uint_as_float((uint32_t)(127 - s) << 23), fsh = __uint_as_float((uint32_t)(127 + s) << 23);
    uint16_t c2;
    asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(c2) : "f"(0.f), "f"(v * ish));
    uint32_t h2;
    asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(h2) : "h"(c2));
    code[pl] = c2 & 0xFFu;
    v -= __half2float(__ushort_as_half((unsigned short)(h2 & 0xFFFFu))) * fsh;
    sc[pl] = (uint32_t)(s + 127);
    sh -= 5;
  }
}

// ---------------------------------------------------------------- E4M3 (OCP FP8, "FN": no infinities)
// Round-to-nearest-even encode of |v| <= 448 (larger magnitudes saturate to
// 448); decode. Written from the format's definition: bias 7, exponent field
// 0 = subnormals m * 2^-9, largest finite 0x7E = 1.75 * 2^8.
__device__ __forceinline__ uint32_t e4m3_encode(float v) {
  const uint32_t s = (__float_as_uint(v) >> 24) & 0x80u;
  const float a = fabsf(v);
  if (!(a > 0.f)) return s;
  if (a >= 448.f) return s | 0x7Eu;
  int e = (int)((__float_as_uint(a) >> 23) & 0xFFu) - 127;
  if (e < -6) {  // subnormal range: multiples of 2^-9 (8 * 2^-9 is the smallest normal, code 0x08)
    const float m = rintf(a * 512.f);
    return s | (uint32_t)m;
  }
  float q = rintf(a * __uint_as_float((uint32_t)(127 - e + 3) << 23));  // a / 2^e * 8 in [8, 16]
  uint32_t mant = (uint32_t)q;
  if (mant == 16u) {
    mant = 8u;
    ++e;
  }
  if (e > 8 || (e == 8 && mant > 14u)) return s | 0x7Eu;
  return s | ((uint32_t)(e + 7) << 3) | (mant - 8u);
}
__device__ __forceinline__ float e4m3_decode(uint32_t b) {
  const uint32_t e = (b >> 3) & 15u, m = b & 7u;
  const float v = e ? __uint_as_float((e + 120u) << 23) * (1.f + 0.125f * (float)m) : (float)m * 0.001953125f;
  return (b & 0x80u) ? -v : v;
}

}  // namespace tc
}  // namespace moe
