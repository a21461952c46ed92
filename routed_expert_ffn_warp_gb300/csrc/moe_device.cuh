// Device primitives shared by the kernels of the routed-expert FFN library:
// MXFP4 fragment decode, m16n8k16 tensor-core MMA, double-float arithmetic,
// and the mbarrier / bulk-copy (TMA) helpers of the streaming pipeline.
#pragma once
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <stdint.h>

#include "../../include/moe.h"
#include "moe_internal.h"

namespace moe {
namespace dev {

// ---------------------------------------------------------------- primitives

__device__ __forceinline__ uint4 ld16(const void* p) { return __ldg(reinterpret_cast<const uint4*>(p)); }
__device__ __forceinline__ uint32_t ld4(const void* p) { return __ldg(reinterpret_cast<const uint32_t*>(p)); }

// Four bytes of E2M1 code pairs to four f16x2 (per byte: low nibble -> low
// half, high nibble -> high half). mov.b32 splits the word into byte registers.
__device__ __forceinline__ void e2m1x8_f16x2(uint32_t w, uint32_t& r0, uint32_t& r1, uint32_t& r2, uint32_t& r3) {
  asm("{\n\t.reg .b8 b0, b1, b2, b3;\n\tmov.b32 {b0, b1, b2, b3}, %4;\n\t"
      "cvt.rn.f16x2.e2m1x2 %0, b0;\n\tcvt.rn.f16x2.e2m1x2 %1, b1;\n\t"
      "cvt.rn.f16x2.e2m1x2 %2, b2;\n\tcvt.rn.f16x2.e2m1x2 %3, b3;\n\t}"
      : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
      : "r"(w));
}

// E8M0 byte to fp32: 2^(e-127); e = 0 is the subnormal 2^-127.
__device__ __forceinline__ float e8m0_f32(uint32_t e) { return __uint_as_float(e ? (e << 23) : 0x00400000u); }

// Four E8M0 bytes to fp32 via two cvt.rn.bf16x2.ue8m0x2 (2^(e-127) is exact in
// bf16, the subnormal 2^-127 included); byte i -> s[i].
__device__ __forceinline__ void e8m0x4_f32(uint32_t w, float (&s)[4]) {
  uint32_t lo, hi;
  const uint16_t w0 = (uint16_t)(w & 0xFFFFu), w1 = (uint16_t)(w >> 16);
  asm("cvt.rn.bf16x2.ue8m0x2 %0, %1;" : "=r"(lo) : "h"(w0));
  asm("cvt.rn.bf16x2.ue8m0x2 %0, %1;" : "=r"(hi) : "h"(w1));
  s[0] = __uint_as_float(lo << 16);
  s[1] = __uint_as_float(lo & 0xFFFF0000u);
  s[2] = __uint_as_float(hi << 16);
  s[3] = __uint_as_float(hi & 0xFFFF0000u);
}

__device__ __forceinline__ void mma16816(float (&d)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1) {
  asm("mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, {%0,%1,%2,%3};\n"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

// A fragments of the two MMAs of scale block bb from a lane's 16 code bytes.
// MMA 1 takes code bytes 4c, 4c+1 of the block (elements 8c..8c+3), MMA 2 bytes
// 4c+2, 4c+3 (elements 8c+4..8c+7); the B fragment is loaded to match.
__device__ __forceinline__ void a_frags(const uint4 q, int bb, uint32_t (&a1)[4], uint32_t (&a2)[4]) {
  const uint32_t rg = bb ? q.z : q.x, rg8 = bb ? q.w : q.y;
  e2m1x8_f16x2(rg, a1[0], a1[2], a2[0], a2[2]);
  e2m1x8_f16x2(rg8, a1[1], a1[3], a2[1], a2[3]);
}

// Gate/up tile: acc[nt] (rows g, g+8 x columns 2c, 2c+1 of n8 tile nt) +=
// sum over the tile's two scale blocks of scale(row, block) * (codes . x16).
template <int NT>
__device__ __forceinline__ void gu_tile(const uint4 q, uint32_t sc, const uint4 (&bx)[NT][2], float (&acc)[NT][4]) {
  float scl[4];
  e8m0x4_f32(sc, scl);
#pragma unroll
  for (int bb = 0; bb < 2; ++bb) {
    uint32_t a1[4], a2[4];
    a_frags(q, bb, a1, a2);
    const float sg = scl[2 * bb];
    const float sg8 = scl[2 * bb + 1];
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) {
      float t[4] = {0.f, 0.f, 0.f, 0.f};
      mma16816(t, a1, bx[nt][bb].x, bx[nt][bb].y);
      mma16816(t, a2, bx[nt][bb].z, bx[nt][bb].w);
      acc[nt][0] = fmaf(t[0], sg, acc[nt][0]);
      acc[nt][1] = fmaf(t[1], sg, acc[nt][1]);
      acc[nt][2] = fmaf(t[2], sg8, acc[nt][2]);
      acc[nt][3] = fmaf(t[3], sg8, acc[nt][3]);
    }
  }
}

// Down tile: columns are (hi, lo) planes of pairs; acc[nt][0|1] = rows g | g+8
// of pair c of tile nt. sb[nt][bb] holds the two per-MMA scales of pair c's h.
template <int NT>
__device__ __forceinline__ void dn_tile(const uint4 q, uint32_t sc, const uint4 (&bh)[NT][2],
                                        const float2 (&sb)[NT][2], float (&acc)[NT][2]) {
  float scl[4];
  e8m0x4_f32(sc, scl);
#pragma unroll
  for (int bb = 0; bb < 2; ++bb) {
    uint32_t a1[4], a2[4];
    a_frags(q, bb, a1, a2);
    const float sg = scl[2 * bb];
    const float sg8 = scl[2 * bb + 1];
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) {
      float t1[4] = {0.f, 0.f, 0.f, 0.f}, t2[4] = {0.f, 0.f, 0.f, 0.f};
      mma16816(t1, a1, bh[nt][bb].x, bh[nt][bb].y);
      mma16816(t2, a2, bh[nt][bb].z, bh[nt][bb].w);
      const float s1 = sb[nt][bb].x, s2 = sb[nt][bb].y;
      acc[nt][0] = fmaf(t1[0] + t1[1], sg * s1, acc[nt][0]);
      acc[nt][0] = fmaf(t2[0] + t2[1], sg * s2, acc[nt][0]);
      acc[nt][1] = fmaf(t1[2] + t1[3], sg8 * s1, acc[nt][1]);
      acc[nt][1] = fmaf(t2[2] + t2[3], sg8 * s2, acc[nt][1]);
    }
  }
}

// Power-of-two exponent sigma with m * 2^sigma in [2^14, 2^15) for m > 0,
// clamped so that both 2^sigma and 2^-sigma are normal fp32 numbers.
__device__ __forceinline__ int f16_headroom_exponent(float m) {
  if (!(m > 0.f)) return 0;
  int ex = (int)((__float_as_uint(m) >> 23) & 0xFFu) - 127;  // floor(log2 m) for normal m
  int s = 14 - ex;
  return s < -112 ? -112 : (s > 126 ? 126 : s);
}
__device__ __forceinline__ float pow2f(int s) { return __uint_as_float((uint32_t)(s + 127) << 23); }

// ---------------------------------------------------------------- double-float helpers
// Error-free transformations (Knuth TwoSum, FMA-based TwoProduct); the _rn
// intrinsics keep the compiler from contracting or reassociating them.
struct dd {
  float hi, lo;
};
__device__ __forceinline__ void two_sum(float a, float b, float& s, float& e) {
  s = __fadd_rn(a, b);
  float bp = __fsub_rn(s, a);
  e = __fadd_rn(__fsub_rn(a, __fsub_rn(s, bp)), __fsub_rn(b, bp));
}
__device__ __forceinline__ void dd_mac(dd& acc, float a, float b) {
  float p = __fmul_rn(a, b);
  float pe = __fmaf_rn(a, b, -p);
  float s, e;
  two_sum(acc.hi, p, s, e);
  acc.hi = s;
  acc.lo = __fadd_rn(acc.lo, __fadd_rn(e, pe));
}
__device__ __forceinline__ dd dd_add(dd a, dd b) {
  float s, e;
  two_sum(a.hi, b.hi, s, e);
  e = __fadd_rn(e, __fadd_rn(a.lo, b.lo));
  dd r;
  r.hi = __fadd_rn(s, e);
  r.lo = __fsub_rn(e, __fsub_rn(r.hi, s));
  return r;
}
__device__ __forceinline__ dd dd_shfl_xor(dd a, int m) {
  dd r;
  r.hi = __shfl_xor_sync(0xffffffffu, a.hi, m);
  r.lo = __shfl_xor_sync(0xffffffffu, a.lo, m);
  return r;
}
// Order-preserving map of a float to an unsigned key (-0 folded into +0): a > b
// as floats iff key(a) > key(b). Every non-NaN float maps above 0x003FFFFF, so
// key 0 can stand for "no candidate". unkey inverts it (+0 for -0).
__device__ __forceinline__ unsigned fkey(float v) {
  const unsigned u = __float_as_uint(v + 0.f);
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}
__device__ __forceinline__ float unkey(unsigned k) {
  return __uint_as_float((k & 0x80000000u) ? (k & 0x7FFFFFFFu) : ~k);
}

// The warp's best candidate: the largest logit (hi, lo) -- hi decides, then lo,
// which for normalised pairs (|lo| <= ulp(hi)/2) is the order of the values --
// then the lowest index, by three redux.sync and no branch: (mh, ml)
// are the winner's keys, the return value its index. A lane without a
// candidate passes keys (0, 0) and index 0x7fffffff.
__device__ __forceinline__ int warp_best_dd(unsigned kh, unsigned kl, int idx, unsigned& mh, unsigned& ml) {
  mh = __reduce_max_sync(0xffffffffu, kh);
  ml = __reduce_max_sync(0xffffffffu, kh == mh ? kl : 0u);
  return (int)__reduce_min_sync(0xffffffffu, (kh == mh && kl == ml) ? (unsigned)idx : 0x7fffffffu);
}

// A lane's running best of its own candidates in the same order, branch-free
// (a divergent branch per candidate costs more than the comparisons).
__device__ __forceinline__ void lane_best_dd(unsigned kh, unsigned kl, int idx, unsigned& bh, unsigned& bl, int& bi) {
  const bool better = kh > bh || (kh == bh && (kl > bl || (kl == bl && idx < bi)));
  bh = better ? kh : bh;
  bl = better ? kl : bl;
  bi = better ? idx : bi;
}


// ---------------------------------------------------------------- mbarrier / bulk copy / timers

__device__ __forceinline__ uint32_t smem_u32(const void* p) { return (uint32_t)__cvta_generic_to_shared(p); }

__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count) : "memory");
}
__device__ __forceinline__ void fence_mbar_init() { asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory"); }
__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\tmbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\tselp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}
// try_wait that may suspend the thread for up to `ns` nanoseconds while the phase is incomplete.
__device__ __forceinline__ bool mbar_try_wait_hint(uint64_t* bar, uint32_t parity, uint32_t ns) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\tmbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n\tselp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity), "r"(ns)
      : "memory");
  return ok != 0;
}
__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}
__device__ __forceinline__ void mbar_arrive_cnt(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)), "r"(count) : "memory");
}
__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)), "r"(bytes) : "memory");
}
// One bulk (TMA, non-tensor) copy global -> this CTA's shared memory; completion
// is signalled on `bar` as transaction bytes. 16-byte aligned, size % 16 == 0.
__device__ __forceinline__ void bulk_g2s(void* dst, const void* src, uint32_t bytes, uint64_t* bar) {
  asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
                   smem_u32(dst)),
               "l"(src), "r"(bytes), "r"(smem_u32(bar))
               : "memory");
}
// Start moving `bytes` (a multiple of 16, 16-byte aligned) at src into L2.
__device__ __forceinline__ void prefetch_l2(const void* src, uint32_t bytes) {
  asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(src), "r"(bytes) : "memory");
}
__device__ __forceinline__ uint64_t globaltimer() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}
__device__ __forceinline__ int ld_acquire(const int* p) {
  int v;
  asm volatile("ld.acquire.gpu.global.b32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}
__device__ __forceinline__ unsigned ld_acquire_u(const unsigned* p) {
  unsigned v;
  asm volatile("ld.acquire.gpu.global.b32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}
__device__ __forceinline__ void st_release_u(unsigned* p, unsigned v) {
  asm volatile("st.release.gpu.global.b32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}
// CTA-scope acquire load / release store of a shared-memory word.
__device__ __forceinline__ int ld_acquire_cta_shared(const int* p) {
  int v;
  asm volatile("ld.acquire.cta.shared::cta.b32 %0, [%1];" : "=r"(v) : "r"(smem_u32(p)) : "memory");
  return v;
}
__device__ __forceinline__ void st_release_cta_shared(int* p, int v) {
  asm volatile("st.release.cta.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(p)), "r"(v) : "memory");
}
__device__ __forceinline__ void named_bar(int id, int threads) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(threads) : "memory");
}
// Named barrier that also ORs a predicate over the participating threads:
// every thread gets the same result.
__device__ __forceinline__ bool named_bar_or(int id, int threads, bool pred) {
  uint32_t r;
  asm volatile(
      "{\n\t.reg .pred p, q;\n\tsetp.ne.u32 p, %1, 0;\n\tbar.red.or.pred q, %2, %3, p;\n\tselp.u32 %0, 1, 0, q;\n\t}"
      : "=r"(r)
      : "r"((uint32_t)pred), "r"(id), "r"(threads)
      : "memory");
  return r != 0;
}
// Generic-proxy writes to global memory <-> later async-proxy (bulk copy) accesses.
__device__ __forceinline__ void fence_proxy_async_global() { asm volatile("fence.proxy.async.global;" ::: "memory"); }
__device__ __forceinline__ uint4 ldcg16(const void* p) { return __ldcg(reinterpret_cast<const uint4*>(p)); }
__device__ __forceinline__ unsigned long long ld_relaxed_u64(const unsigned long long* p) {
  unsigned long long v;
  asm volatile("ld.relaxed.gpu.global.b64 %0, [%1];" : "=l"(v) : "l"(p) : "memory");
  return v;
}
__device__ __forceinline__ void ld_relaxed_u64x2(const unsigned long long* p, unsigned long long& a,
                                                 unsigned long long& b) {
  asm volatile("ld.relaxed.gpu.global.v2.u64 {%0, %1}, [%2];" : "=l"(a), "=l"(b) : "l"(p) : "memory");
}
__device__ __forceinline__ void st_relaxed_u64(unsigned long long* p, unsigned long long v) {
  asm volatile("st.relaxed.gpu.global.b64 [%0], %1;" ::"l"(p), "l"(v) : "memory");
}

// ---------------------------------------------------------------- cp.async streams and MMA helpers

__device__ __forceinline__ void cp16(void* dst, const void* src) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(smem_u32(dst)), "l"(src) : "memory");
}
__device__ __forceinline__ void cp_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_wait() {
  asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}
__device__ __forceinline__ void cp_wait_all() { asm volatile("cp.async.wait_all;" ::: "memory"); }
// Arrive on `bar` once all of this thread's earlier cp.async copies have landed.
__device__ __forceinline__ void cp_arrive(uint64_t* bar) {
  asm volatile("cp.async.mbarrier.arrive.noinc.shared::cta.b64 [%0];" ::"r"(smem_u32(bar)) : "memory");
}

// Bounded wait for a staged chunk (its copies always land; the bound only
// guarantees that no wait can hang): on expiry the status word says timeout.
__device__ __forceinline__ void wait_chunk(uint64_t* bar, uint32_t parity, int* status) {
  if (mbar_try_wait(bar, parity)) return;
  const uint64_t t0 = globaltimer();
  while (!mbar_try_wait(bar, parity)) {
    if ((long long)(globaltimer() - t0) > 50000000LL) {
      atomicCAS(status, 0, MOE_ERR_TIMEOUT);
      return;
    }
  }
}

// D = A * B (no accumulator input).
__device__ __forceinline__ void mma_z(float (&d)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1) {
  asm("mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
      "{%10,%10,%10,%10};\n"
      : "=f"(d[0]), "=f"(d[1]), "=f"(d[2]), "=f"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1), "f"(0.f));
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

// Programmatic dependent launch: wait for the preceding grid / let the next one launch.
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_launch_dependents() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }
// First statement of every kernel of the forward chain: nothing before it
// touches global memory, so the kernel sees all writes of the grids before it
// (each of which waited the same way); the next grid may then be scheduled and
// sits in its own wait, which hides its launch behind this grid's work. At most
// two grids of the chain are resident at a time, and only the running one
// holds tensor memory.
__device__ __forceinline__ void pdl_enter() {
  pdl_wait();
  pdl_launch_dependents();
}

}  // namespace dev
}  // namespace moe
