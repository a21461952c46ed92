// Fused decode path: the whole MoE layer for T <= 16 tokens in ONE persistent
// kernel, one CTA per SM, 16 warps.
//
//   A  x is staged in shared memory; CTA b computes the double-float router
//      logits of experts b, b+G, ... from it and publishes each as two 64-bit
//      words (value bits | launch sequence number); x is then scaled to f16 in
//      place (for T <= 8 by spare warps during phase B's poll).
//   B  token warps poll the published words of all experts (a dataflow
//      barrier: no grid-wide sync, no atomics), then every CTA redundantly runs
//      top-k + softmax gates, the counting sort of the T*k pairs and the slot
//      list (identical, deterministic results in every CTA).
//   C  gate/up units (slot, 16-row pair tile) are split evenly over the CTAs,
//      and each unit's k tiles into 3 fixed chunks (a split that depends on the
//      unit alone, so its sums do not depend on the batch). A CTA's chunks are
//      dealt to its 16 warps round-robin. Every warp streams its own chunks
//      through a private shared-memory ring with cp.async (16-byte copies, no
//      L1), several KB ahead of its math, so no warp waits on another for
//      data. The last of a unit's 3 chunk warps to finish adds the 3 partial
//      sums in chunk order, applies SiLU(gate)*up and publishes h (f16 hi +
//      lo with a power-of-two scale per 16 elements) as 64-bit words that
//      carry the launch sequence number, like the logits.
//   D  down units (slot, token half of <= 8 tokens, 16 output rows) in that
//      order, chunked and dealt the same way; each warp's down tiles follow
//      its gate/up tiles in its ring. For each (slot, half) of the CTA the
//      CTA stages the slot's h in shared memory, polling (bounded) the words
//      until they carry this launch's number;
//      the last chunk warp of a unit publishes its partial rows as tagged
//      words, and the warp holding a row tile's unit of the last (slot, half)
//      combines the tile once every pair's words carry this launch's number:
//      y = sum_j g_j part_j (top-k order j) + shared, one rounding.
//
// The pages: expert pairs grouped by expert, one pass over each selected
// expert's rows for all of its tokens, fused gate/up then down, a row summed
// over all of a token's experts in a fixed order ("NInfer" Qwen3.8-Flash-Next
// notes, MoE execution bullets); per-layer work replayed as a CUDA graph
// ("Neural Server" technical page, "How one token and one prompt are
// processed").
//
// Every device-side wait is bounded (%globaltimer); on expiry the CTA records
// MOE_ERR_TIMEOUT in the status word, stops waiting, and runs to completion,
// so no wait can hang the GPU. All CTAs must be co-resident: the grid is one
// CTA per SM and every CTA needs more than half of an SM's shared memory;
// contexts use this kernel only when the occupancy API says one CTA fits on
// an SM. A GPU shared with another context that holds SMs can still keep a
// CTA waiting: its waits then give up and the status word reports it.
#include <stdint.h>

#include <algorithm>

#include "../../include/moe.h"
#include "moe_device.cuh"
#include "moe_fused_route.cuh"
#include "moe_internal.h"

namespace moe {
namespace {

using namespace dev;

constexpr int kChunks = 3;         // fixed k-tile chunks of every unit
constexpr int kHalf = 8;           // tokens of a down unit (a slot with more tokens has two halves)
constexpr int kGroupBytes = 2 * kTileBytes;  // a ring slot: one gate/up tile pair or two down tiles
constexpr int kMaxUS = 8;                       // unit slots (partial-sum buffers) per phase, at most
constexpr int kRing = 4;                        // groups in each warp's weight ring

__device__ __forceinline__ Shared carve(uint8_t* sm, const DecParams& p) {
  Shared s;
  s.ctl = reinterpret_cast<int*>(sm);
  s.x16 = reinterpret_cast<__half*>(sm + p.off_x16);
  s.hst = s.x16;
  s.hsc = reinterpret_cast<float*>(sm + p.off_hsc);
  s.xinv = reinterpret_cast<float*>(sm + p.off_xinv);
  s.red = reinterpret_cast<dd*>(sm + p.off_red);
  s.pgu = reinterpret_cast<float*>(sm + p.off_pgu);
  s.pdn = reinterpret_cast<float*>(sm + p.off_pdn);
  carve_route(s, sm, p);
  s.ring = sm + p.off_ring;
  return s;
}

// ---------------------------------------------------------------- work units

struct Unit {
  int slot, idx, e, q0, n, f;  // q0, n: first h/part row and rows (tokens) of the unit
};

__device__ __forceinline__ Unit gu_unit(const DecParams& p, const Shared& s, int u) {
  const int nr = s.misc[0];
  const int uf = p.f.F / 16;
  Unit r;
  if (u < nr * uf) {
    r.slot = u / uf;
    r.idx = u - r.slot * uf;
    r.f = p.f.F;
  } else {
    r.slot = nr;
    r.idx = u - nr * uf;
    r.f = p.f.S;
  }
  r.e = s.slot_e[r.slot];
  r.q0 = s.slot_q0[r.slot];
  r.n = s.slot_n[r.slot];
  return r;
}

// Down unit u: (slot, half) pair u / (d/16), row tile u % (d/16).
__device__ __forceinline__ Unit dn_unit(const DecParams& p, const Shared& s, int u) {
  const int ud = p.f.d / 16;
  const int hs = u / ud;
  Unit r;
  r.slot = s.hs_slot[hs];
  r.idx = u - hs * ud;
  const int half = s.hs_half[hs];
  r.e = s.slot_e[r.slot];
  r.q0 = s.slot_q0[r.slot] + kHalf * half;
  r.n = min(kHalf, s.slot_n[r.slot] - kHalf * half);
  r.f = (r.e == p.f.E) ? p.f.S : p.f.F;
  return r;
}

__device__ __forceinline__ int token_of(const DecParams& p, const Shared& s, int q) {
  return q < p.f.P ? s.perm[q] / p.f.k : q - p.f.P;
}

__device__ __forceinline__ void unit_range(int total, int& b0, int& b1) {
  b0 = (int)(((long long)blockIdx.x * total) / gridDim.x);
  b1 = (int)(((long long)(blockIdx.x + 1) * total) / gridDim.x);
}

// k-tile range [k0, k1) of chunk c of a unit with K64 k tiles.
__device__ __forceinline__ void chunk_range(int K64, int c, int& k0, int& k1) {
  const int ck = (K64 + kChunks - 1) / kChunks;
  k0 = min(K64, c * ck);
  k1 = min(K64, k0 + ck);
}

// Staged x row t (bf16, in place) -> f16 * 2^sigma_t by one warp; K padding zeroed.
__device__ void scale_x_token(const DecParams& p, const Shared& s, int t) {
  const FwdParams& f = p.f;
  const int lane = threadIdx.x & 31;
  const int d8 = f.d / 8;
  {
    uint4* xr = reinterpret_cast<uint4*>(s.x16 + (size_t)t * p.xstride);
    float m = 0.f;
    for (int o = lane; o < d8; o += 32) {
      const uint4 v = xr[o];
      const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
      for (int j = 0; j < 4; ++j)
        m = fmaxf(m, fmaxf(fabsf(__uint_as_float(w[j] << 16)), fabsf(__uint_as_float(w[j] & 0xFFFF0000u))));
    }
    for (int o = 16; o; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
    const int sg = f16_headroom_exponent(m);
    const float sc = pow2f(sg);
    for (int o = lane; o < d8; o += 32) {
      const uint4 v = xr[o];
      const uint32_t w[4] = {v.x, v.y, v.z, v.w};
      uint32_t h[4];
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const __half2 hv =
            __floats2half2_rn(__uint_as_float(w[j] << 16) * sc, __uint_as_float(w[j] & 0xFFFF0000u) * sc);
        h[j] = *reinterpret_cast<const uint32_t*>(&hv);
      }
      xr[o] = make_uint4(h[0], h[1], h[2], h[3]);
    }
    for (int o = d8 + lane; o < f.d64 / 8; o += 32) xr[o] = make_uint4(0, 0, 0, 0);
    if (lane == 0) s.xinv[t] = pow2f(-sg);
  }
}

// All tokens, one warp per token.
__device__ void scale_x(const DecParams& p, const Shared& s) {
  for (int t = threadIdx.x >> 5; t < p.f.T; t += kWarps) scale_x_token(p, s, t);
}

// With T <= kWarps / 2 the x scaling runs on warps kWarps-1, kWarps-2, ...
// while warps 0 .. T-1 poll the logit words and take the top k.
__device__ __forceinline__ bool scale_x_beside_topk(const DecParams& p) { return p.f.T <= kWarps / 2; }

// The (slot, half) pairs of the down phase, in slot order: a slot with more
// than kHalf tokens contributes two (tokens [0, 8) and [8, n)). One warp,
// after the whole CTA's sort of more than 32 pairs (the small sort lists them
// itself).
__device__ void build_halves(const Shared& s) {
  const int lane = threadIdx.x & 31;
  const int nsl = s.misc[1], nr = s.misc[0];
  int base = 0, routed = 0;
  for (int s0 = 0; s0 < nsl; s0 += 32) {
    const int sl = s0 + lane;
    const int h = sl < nsl ? (s.slot_n[sl] > kHalf ? 2 : 1) : 0;
    int inc = h;
    for (int o = 1; o < 32; o <<= 1) {
      const int v = __shfl_up_sync(0xffffffffu, inc, o);
      if (lane >= o) inc += v;
    }
    for (int j = 0; j < h; ++j) {
      s.hs_slot[base + inc - h + j] = sl;
      s.hs_half[base + inc - h + j] = j;
    }
    routed += (int)__reduce_add_sync(0xffffffffu, (unsigned)(sl < nr ? h : 0));
    base += __shfl_sync(0xffffffffu, inc, 31);
  }
  if (lane == 0) {
    s.misc[4] = base;
    s.misc[5] = routed;
  }
}

// kSmall: the instantiation for E <= 128, at most 4 tokens and 32 pairs (the
// decode shape) carries only the code those calls run: a third less code to
// fetch into cold instruction caches every launch (measured 0.25 us per layer).
template <bool kSmall>
__device__ void routing(const DecParams& p, const Shared& s, unsigned seq, volatile int* abort) {
  const int warp = threadIdx.x >> 5;
  if (warp < p.f.T) {
    if (kSmall || p.f.E <= 128) topk_token<4>(p, s, warp, seq, abort);
    else if (p.f.E <= 256) topk_token<8>(p, s, warp, seq, abort);
    else topk_token<16>(p, s, warp, seq, abort);
  } else if (scale_x_beside_topk(p) && warp >= kWarps - p.f.T) {
    scale_x_token(p, s, kWarps - 1 - warp);
  }
  __syncthreads();
  if (!kSmall && p.f.P > 32) {  // the whole CTA sorts
    bucket_large(p, s);
    __syncthreads();
  }
  if (warp == 0) {
    if (kSmall || p.f.P <= 32) {
      bucket_small<kHalf>(p, s);
    } else {
      __syncwarp();
      build_halves(s);
    }
  } else if (warp == 1 && blockIdx.x == 0 && p.f.P <= 32) {
    export_counts_small(p, s);
  }
  __syncthreads();
}

// ---------------------------------------------------------------- phases C + D: per-warp weight streams
//
// The CTA's items (unit, chunk) -- its gate/up items, then its down items --
// are dealt to the 16 warps round-robin (item i to warp i % 16). A warp copies
// the weight tiles of its items, in order, through its own ring of RG slots of
// 1,088 bytes (a gate/up tile pair, or two consecutive down tiles) with
// cp.async, RG slots ahead of the math; completion
// is tracked with per-thread cp.async groups (one group per slot, empty groups
// past the end of the stream keep the count uniform).

__device__ __forceinline__ void cp_async16(void* dst, const void* src, uint64_t pol) {
#ifndef MOE_NO_L2_HINT
  asm volatile("cp.async.cg.shared.global.L2::cache_hint [%0], [%1], 16, %2;" ::"r"(smem_u32(dst)), "l"(src),
               "l"(pol)
               : "memory");
#else
  (void)pol;
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(smem_u32(dst)), "l"(src) : "memory");
#endif
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
__device__ __forceinline__ void cp_async_wait_all() { asm volatile("cp.async.wait_all;" ::: "memory"); }
// Wait until at most N of this thread's most recent groups are pending.
template <int N>
__device__ __forceinline__ void cp_async_wait() {
  asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}
// L2 policy for the weight stream: each byte is read once per layer call.
__device__ __forceinline__ uint64_t evict_first_policy() {
  uint64_t pol;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(pol));
  return pol;
}

// The CTA's work: its ranges of gate/up and down units.
struct Plan {
  int g0, ngu;  // gate/up units [g0, g0 + ngu)
  int d0, ndn;  // down units [d0, d0 + ndn)
  int nguw, ndnw;  // items of this warp in each phase
};

__device__ __forceinline__ int warp_items(int n_items, int w) { return n_items > w ? (n_items - w + kWarps - 1) / kWarps : 0; }

__device__ __forceinline__ Plan make_plan(const DecParams& p, const Shared& s, int w) {
  const FwdParams& f = p.f;
  const int NUg = s.misc[0] * (f.F / 16) + (s.misc[1] > s.misc[0] ? f.S / 16 : 0);  // + the shared slot, if any
  const int NUd = s.misc[4] * (f.d / 16);
  Plan pl;
  int b1;
  unit_range(NUg, pl.g0, b1);
  pl.ngu = b1 - pl.g0;
  unit_range(NUd, pl.d0, b1);
  pl.ndn = b1 - pl.d0;
  pl.nguw = warp_items(kChunks * pl.ngu, w);
  pl.ndnw = warp_items(kChunks * pl.ndn, w);
  return pl;
}

// Item j of warp w: CTA-local unit, chunk, k-tile range, source of its first
// group, and its groups.
struct Item {
  int u;     // CTA-local unit index within its phase
  int c;     // chunk
  int k0, k1;
  bool down;
  const uint8_t* src;
  int ng;         // slots (groups) of the item
  int last_bytes; // bytes of its last group
};

__device__ __forceinline__ Item item_of(const DecParams& p, const Shared& s, const Plan& pl, int w, int j) {
  const FwdParams& f = p.f;
  Item it;
  if (j < pl.nguw) {
    const int i = w + kWarps * j;
    it.u = i / kChunks;
    it.c = i - it.u * kChunks;
    it.down = false;
    const Unit un = gu_unit(p, s, pl.g0 + it.u);
    const int K64d = k64_tiles(f.d);
    chunk_range(K64d, it.c, it.k0, it.k1);
    it.src = f.packed + (size_t)weight_index(f, un.e) * f.expert_stride + ((size_t)un.idx * K64d + it.k0) * kGroupBytes;
    it.ng = it.k1 - it.k0;
    it.last_bytes = kGroupBytes;
  } else {
    const int i = w + kWarps * (j - pl.nguw);
    it.u = i / kChunks;
    it.c = i - it.u * kChunks;
    it.down = true;
    const Unit un = dn_unit(p, s, pl.d0 + it.u);
    const int K64f = k64_tiles(un.f);
    chunk_range(K64f, it.c, it.k0, it.k1);
    it.src = f.packed + (size_t)weight_index(f, un.e) * f.expert_stride + gu_packed_bytes(f.d, un.f) +
             ((size_t)un.idx * K64f + it.k0) * kTileBytes;
    const int nt = it.k1 - it.k0;
    it.ng = (nt + 1) / 2;
    it.last_bytes = (nt & 1) ? kTileBytes : kGroupBytes;
  }
  return it;
}

// Issue cursor of a warp's stream.
struct Cursor {
  int j, g, ng, nitems, last_bytes;
  const uint8_t* src;
};

__device__ __forceinline__ void cursor_seek(const DecParams& p, const Shared& s, const Plan& pl, int w, Cursor& cu) {
  while (cu.j < cu.nitems) {
    const Item it = item_of(p, s, pl, w, cu.j);
    if (it.ng > 0) {
      cu.src = it.src;
      cu.ng = it.ng;
      cu.last_bytes = it.last_bytes;
      cu.g = 0;
      return;
    }
    ++cu.j;
  }
}

// Copy the cursor's next group into ring slot `dst` (one cp.async group; an
// empty group once the stream is exhausted) and advance.
__device__ __forceinline__ void issue_group(const DecParams& p, const Shared& s, const Plan& pl, int w, Cursor& cu,
                                            uint8_t* dst, uint64_t pol) {
  const int lane = threadIdx.x & 31;
  if (cu.j < cu.nitems) {
    const int n16 = (cu.g == cu.ng - 1 ? cu.last_bytes : kGroupBytes) / 16;
    for (int k = lane; k < n16; k += 32) cp_async16(dst + 16 * k, cu.src + 16 * k, pol);
    cu.src += kGroupBytes;
    if (++cu.g == cu.ng) {
      ++cu.j;
      cursor_seek(p, s, pl, w, cu);
    }
  }
  cp_async_commit();
}

// Per-unit partial-sum slots: writers of CTA-local unit u use slot u % n_us
// once its owner word says u; the reducer hands the slot to unit u + n_us.
__device__ bool claim_slot(const DecParams& p, int* owner, int u, volatile int* abort) {
  int ok = 1;
  if ((threadIdx.x & 31) == 0 && ld_acquire_cta_shared(owner) != u) {
    const uint64_t t0 = globaltimer();
    while (ld_acquire_cta_shared(owner) != u) {
      if (*abort || timed_out(t0, p.wait_ns)) {
        if (!*abort) give_up(abort, p.f.status);
        ok = 0;
        break;
      }
    }
  }
  ok = __shfl_sync(0xffffffffu, ok, 0);
  __syncwarp();
  return ok != 0;
}

// Count this warp's chunk of unit slot `us`; true for the last of the 3.
__device__ __forceinline__ bool arrive_chunk(int* arrivals) {
  __syncwarp();
  int last = 0;
  if ((threadIdx.x & 31) == 0) {
    __threadfence_block();
    last = atomicAdd(arrivals, 1) == kChunks - 1;
    if (last) __threadfence_block();
  }
  last = __shfl_sync(0xffffffffu, last, 0);
  __syncwarp();
  return last != 0;
}

__device__ __forceinline__ void free_slot(int* arrivals, int* owner, int next_owner) {
  __syncwarp();
  if ((threadIdx.x & 31) == 0) {
    *arrivals = 0;
    st_release_cta_shared(owner, next_owner);
  }
}

// Gate/up unit epilogue (the last chunk warp): h for the 16 rows S_tau of the
// unit and each of its tokens. Lanes 0-15 take rows 0-15 of an even token,
// lanes 16-31 of the next one; the f16 scale of h is shared by a token's 16 rows.
__device__ void gateup_reduce(const DecParams& p, const Shared& s, const Unit& un, const float* pb) {
  const FwdParams& f = p.f;
  const unsigned seq = (unsigned)s.misc[3];
  const int lane = threadIdx.x & 31, r = lane & 15;
  const int tc = p.tcap, cs = 32 * tc;  // chunk stride
  for (int m0 = 0; m0 < un.n; m0 += 2) {
    const int m = m0 + (lane >> 4);
    float h = 0.f;
    if (m < un.n) {
      float gs = 0.f, us = 0.f;
#pragma unroll
      for (int c = 0; c < kChunks; ++c) {
        gs += pb[c * cs + r * tc + m];
        us += pb[c * cs + (16 + r) * tc + m];
      }
      const float xi = s.xinv[token_of(p, s, un.q0 + m)];
      const float gate = gs * xi, up = us * xi;
      h = gate / (1.f + expf(-gate)) * up;
    }
    float mx = fabsf(h);
    for (int o = 1; o < 16; o <<= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
    if (m < un.n) {
      const int sh = f16_headroom_exponent(mx);
      const int q = un.q0 + m;
      const int i = 32 * (un.idx >> 1) + 8 * (r >> 2) + 4 * (un.idx & 1) + (r & 3);
      const float v = h * pow2f(sh);
      const __half vh = __float2half_rn(v);
      const __half vl = __float2half_rn(v - __half2float(vh));
      // each value travels with this launch's number: the readers poll the data itself
      const uint32_t hl = (uint32_t)__half_as_ushort(vh) | ((uint32_t)__half_as_ushort(vl) << 16);
      st_relaxed_u64(p.hwords + (size_t)q * f.fmax64 + i, ((unsigned long long)hl << 32) | seq);
      if (r == 0)
        st_relaxed_u64(p.hswords + (size_t)q * f.hgroups + un.idx,
                       ((unsigned long long)__float_as_uint(pow2f(-sh)) << 32) | seq);
    }
  }
}

// Down unit epilogue (the last chunk warp): the unit's 16 partial rows of each
// of its tokens, published as 64-bit words that carry the launch sequence
// number (payload fp32 bits << 32), like h: the combining CTA polls the data.
__device__ void down_reduce(const DecParams& p, const Shared& s, const Unit& un, const float* pb) {
  const FwdParams& f = p.f;
  const unsigned seq = (unsigned)s.misc[3];
  const int lane = threadIdx.x & 31;
  const int hh = min(kHalf, p.tcap), cs = 16 * hh;
  for (int o = lane; o < 16 * un.n; o += 32) {
    const int r = o & 15, m = o >> 4;
    float a = 0.f;
#pragma unroll
    for (int c = 0; c < kChunks; ++c) a += pb[c * cs + r * hh + m];
    st_relaxed_u64(p.pwords + (size_t)(un.q0 + m) * f.d + 16 * un.idx + r,
                   ((unsigned long long)__float_as_uint(a) << 32) | seq);
  }
}

// Wait (bounded) until each of the n words at w[i] carries launch number seq
// in its low half, reloading all the stale ones together; v[i] holds them.
// A null w[i] counts as present.
template <int N>
__device__ __forceinline__ void poll_words(const DecParams& p, const unsigned long long* const (&w)[N],
                                           unsigned long long (&v)[N], unsigned seq, volatile int* abort) {
#pragma unroll
  for (int i = 0; i < N; ++i) v[i] = w[i] ? ld_relaxed_u64(w[i]) : (unsigned long long)seq;
  uint64_t t0 = 0;
  while (true) {
    bool stale = false;
#pragma unroll
    for (int i = 0; i < N; ++i) stale = stale || (unsigned)v[i] != seq;
    if (!stale || *abort) return;
    if (t0 == 0) t0 = globaltimer();
    else if (timed_out(t0, p.wait_ns)) {
      give_up(abort, p.f.status);
      return;
    }
#pragma unroll
    for (int i = 0; i < N; ++i)
      if ((unsigned)v[i] != seq) v[i] = ld_relaxed_u64(w[i]);
  }
}

// Row tile idx of every token, by the CTA that runs the tile's down unit of
// the last (slot, half) pair: y = sum_j g_j part_j (the token's pairs in
// top-k order; pairs of other shards add 0) + shared, one rounding. The
// partial rows come from the tile's down units in other CTAs as tagged words:
// no fence, no counter, one round trip once they are all written.
__device__ void combine_rows(const DecParams& p, const Shared& s, int idx, volatile int* abort) {
  const FwdParams& f = p.f;
  const unsigned seq = (unsigned)s.misc[3];
  const int lane = threadIdx.x & 31;
  const int r0 = 16 * idx, n = f.T * 16;
  constexpr int kJ = 8;  // pairs whose words are in flight together
  for (int o = lane; o < n; o += 32) {
    const int t = o >> 4, r = o & 15;
    float a = 0.f;
    for (int j0 = 0; j0 < f.k; j0 += kJ) {  // sums kept in top-k order
      const unsigned long long* w[kJ];
      unsigned long long v[kJ];
#pragma unroll
      for (int jj = 0; jj < kJ; ++jj) {
        const int j = j0 + jj;
        w[jj] = (j < f.k && expert_in_shard(s.ids[t * f.k + j], f.e_begin, f.e_end))
                    ? p.pwords + (size_t)s.inv[t * f.k + j] * f.d + r0 + r
                    : nullptr;  // this shard's pairs only (all of them without sharding)
      }
      poll_words<kJ>(p, w, v, seq, abort);
#pragma unroll
      for (int jj = 0; jj < kJ; ++jj)
        if (j0 + jj < f.k) a = fmaf(s.gates[t * f.k + j0 + jj], w[jj] ? __uint_as_float((unsigned)(v[jj] >> 32)) : 0.f, a);
    }
    float y = a;
    if (f.S > 0 && f.e_begin == 0) {
      const unsigned long long* w[1] = {p.pwords + (size_t)(f.P + t) * f.d + r0 + r};
      unsigned long long v[1];
      poll_words<1>(p, w, v, seq, abort);
      y += (f.w_sg ? s.sg[t] : 1.f) * __uint_as_float((unsigned)(v[0] >> 32));
    }
    if (f.out_f32) reinterpret_cast<float*>(f.out)[(size_t)t * f.d + r0 + r] = y;
    else reinterpret_cast<__nv_bfloat16*>(f.out)[(size_t)t * f.d + r0 + r] = __float2bfloat16_rn(y);
  }
}

// Stage h of (slot, half) pair hs in shared memory (all threads, after every
// warp is done reading the shared x, which this area overlays): planes
// [m][hi | lo][hstride] and the per-16 scales. The gate/up reducers publish
// h and its scales as 64-bit words (payload << 32 | launch number), so the
// staging loads poll the data itself: no counter, no fence on either side.
// Padding past the slot's ffn is zero.
__device__ void stage_h(const DecParams& p, const Shared& s, int hs, volatile int* abort) {
  const FwdParams& f = p.f;
  const unsigned seq = (unsigned)s.misc[3];
  const int slot = s.hs_slot[hs], half = s.hs_half[hs];
  const int q0 = s.slot_q0[slot] + kHalf * half, n = min(kHalf, s.slot_n[slot] - kHalf * half);
  const int fsl = (s.slot_e[slot] == f.E) ? f.S : f.F;
  // Scale words and h words. Each round, every thread first issues all of its
  // loads (kB of each), then reloads every word that does not yet carry this
  // launch's number, all of them together, until none is stale (bounded): one
  // round trip per retry, not one per word. The timeout test makes the scale
  // words wait for a number no launch writes.
  constexpr int kB = 4;
  const unsigned want_sc = seq + (unsigned)p.test_extra;
  const long long lim = p.test_extra ? p.test_wait_ns : p.wait_ns;
  const int per_row = f.fmax64 / 2;  // element pairs of a row
  const int nsc = n * f.hgroups, nh = n * per_row, per_round = kThreads * kB;
  const int rounds = (max(nsc, nh) + per_round - 1) / per_round;
  for (int rd = 0; rd < rounds; ++rd) {
    const int o0 = rd * per_round + threadIdx.x;
    unsigned long long v[kB], a[kB], b[kB];
    const unsigned long long* wsc[kB];
    const unsigned long long* wh[kB];
#pragma unroll
    for (int u = 0; u < kB; ++u) {
      const int o = o0 + u * kThreads;
      const int ms = o / f.hgroups, k = o - ms * f.hgroups;
      const int m = o / per_row, i = 2 * (o - m * per_row);
      wsc[u] = (o < nsc && 16 * k < fsl) ? p.hswords + (size_t)(q0 + ms) * f.hgroups + k : nullptr;
      wh[u] = (o < nh && i < fsl) ? p.hwords + (size_t)(q0 + m) * f.fmax64 + i : nullptr;
      v[u] = wsc[u] ? ld_relaxed_u64(wsc[u]) : (unsigned long long)want_sc;
      a[u] = b[u] = (unsigned long long)seq;
      if (wh[u]) ld_relaxed_u64x2(wh[u], a[u], b[u]);
    }
    uint64_t t0 = 0;
    while (true) {
      bool stale = false;
#pragma unroll
      for (int u = 0; u < kB; ++u)
        stale = stale || (unsigned)v[u] != want_sc || (unsigned)a[u] != seq || (unsigned)b[u] != seq;
      if (!stale || *abort) break;
      if (t0 == 0) t0 = globaltimer();
      else if (timed_out(t0, lim)) {
        give_up(abort, f.status);
        break;
      }
#pragma unroll
      for (int u = 0; u < kB; ++u) {
        if ((unsigned)v[u] != want_sc) v[u] = ld_relaxed_u64(wsc[u]);
        if ((unsigned)a[u] != seq || (unsigned)b[u] != seq) ld_relaxed_u64x2(wh[u], a[u], b[u]);
      }
    }
    const bool ok = !*abort;
#pragma unroll
    for (int u = 0; u < kB; ++u) {
      const int o = o0 + u * kThreads;
      if (o < nsc) {
        const int ms = o / f.hgroups, k = o - ms * f.hgroups;
        s.hsc[ms * f.hgroups + k] = (wsc[u] && ok) ? __uint_as_float((unsigned)(v[u] >> 32)) : 0.f;
      }
      if (o < nh) {
        const int m = o / per_row, i = 2 * (o - m * per_row);
        uint32_t hv = 0, lv = 0;  // two f16 of each plane
        if (wh[u] && ok) {
          const uint32_t pa = (uint32_t)(a[u] >> 32), pb = (uint32_t)(b[u] >> 32);
          hv = (pa & 0xFFFFu) | (pb << 16);
          lv = (pa >> 16) | (pb & 0xFFFF0000u);
        }
        *reinterpret_cast<uint32_t*>(s.hst + (size_t)(m * 2) * p.hstride + i) = hv;
        *reinterpret_cast<uint32_t*>(s.hst + (size_t)(m * 2 + 1) * p.hstride + i) = lv;
      }
    }
  }
}

template <int NT>
__device__ __forceinline__ void gateup_group(const DecParams& p, const Shared& s, const uint8_t* slot, int kt,
                                             const int (&tokB)[NT], float (&acc)[2 * NT * 4]) {
  const int lane = threadIdx.x & 31, g = lane >> 2, c = lane & 3;
  const uint4 qg = *reinterpret_cast<const uint4*>(slot + 16 * lane);
  const uint32_t sgv = *reinterpret_cast<const uint32_t*>(slot + kTileCodeBytes + 4 * g);
  const uint4 qu = *reinterpret_cast<const uint4*>(slot + kTileBytes + 16 * lane);
  const uint32_t suv = *reinterpret_cast<const uint32_t*>(slot + kTileBytes + kTileCodeBytes + 4 * g);
  uint4 bx[NT][2];
#pragma unroll
  for (int nt = 0; nt < NT; ++nt)
#pragma unroll
    for (int bb = 0; bb < 2; ++bb)
      bx[nt][bb] = tokB[nt] >= 0 ? *reinterpret_cast<const uint4*>(s.x16 + (size_t)tokB[nt] * p.xstride + kt * 64 +
                                                                   bb * 32 + c * 8)
                                 : make_uint4(0, 0, 0, 0);
  float (&ag)[NT][4] = *reinterpret_cast<float(*)[NT][4]>(acc);
  float (&au)[NT][4] = *reinterpret_cast<float(*)[NT][4]>(acc + NT * 4);
  gu_tile<NT>(qg, sgv, bx, ag);
  gu_tile<NT>(qu, suv, bx, au);
}

template <int NT>
__device__ __forceinline__ void down_tile_smem(const DecParams& p, const Shared& s, const uint8_t* t8, int kt,
                                               int nh, float (&acc)[NT][2]) {
  const int lane = threadIdx.x & 31, g = lane >> 2, c = lane & 3;
  const uint4 q = *reinterpret_cast<const uint4*>(t8 + 16 * lane);
  const uint32_t scv = *reinterpret_cast<const uint32_t*>(t8 + kTileCodeBytes + 4 * g);
  uint4 bh[NT][2];
  float2 sb[NT][2];
#pragma unroll
  for (int nt = 0; nt < NT; ++nt) {
    const int mb = 4 * nt + (g >> 1), md = 4 * nt + c;
#pragma unroll
    for (int bb = 0; bb < 2; ++bb) {
      bh[nt][bb] = mb < nh ? *reinterpret_cast<const uint4*>(s.hst + (size_t)(mb * 2 + (g & 1)) * p.hstride +
                                                             kt * 64 + bb * 32 + c * 8)
                           : make_uint4(0, 0, 0, 0);
      sb[nt][bb] = md < nh ? *reinterpret_cast<const float2*>(s.hsc + md * p.f.hgroups + 2 * (2 * kt + bb))
                           : make_float2(0.f, 0.f);
    }
  }
  dn_tile<NT>(q, scv, bh, sb, acc);
}

// Consume the groups of one item from the warp's ring (kc: the warp's count
// of consumed groups; every consumed slot is refilled from the cursor).
template <int NT, int RG>
__device__ void gateup_item(const DecParams& p, const Shared& s, const Plan& pl, const Item& it, const Unit& un,
                            uint8_t* ring, int& slot, Cursor& cu, uint64_t pol, int w, volatile int* abort) {
  const int lane = threadIdx.x & 31, g = lane >> 2, c = lane & 3;
  float acc[2 * NT * 4];
#pragma unroll
  for (int i = 0; i < 2 * NT * 4; ++i) acc[i] = 0.f;
  int tokB[NT];
#pragma unroll
  for (int nt = 0; nt < NT; ++nt) {
    const int m = 8 * nt + g;
    tokB[nt] = (m < un.n) ? token_of(p, s, un.q0 + m) : -1;
  }
  for (int kt = it.k0; kt < it.k1; ++kt) {
    cp_async_wait<RG - 1>();
    __syncwarp();
    uint8_t* sl = ring + slot * kGroupBytes;
    gateup_group<NT>(p, s, sl, kt, tokB, acc);
    __syncwarp();
    issue_group(p, s, pl, w, cu, sl, pol);
    if (++slot == RG) slot = 0;
  }
  const int us = it.u % p.n_us;
  if (!claim_slot(p, s.ctl + kMaxUS + us, it.u, abort)) return;
  float* pb = s.pgu + (size_t)us * kChunks * 32 * p.tcap;
  {
    float* pw = pb + it.c * 32 * p.tcap;  // [gate | up][16 rows][tcap columns]
    const int tc = p.tcap;
#pragma unroll
    for (int nt = 0; nt < NT; ++nt)
#pragma unroll
      for (int r = 0; r < 4; ++r) {
        const int row = g + 8 * (r >> 1), col = 8 * nt + 2 * c + (r & 1);
        if (col < un.n) {
          pw[row * tc + col] = acc[nt * 4 + r];
          pw[(16 + row) * tc + col] = acc[NT * 4 + nt * 4 + r];
        }
      }
  }
  if (!arrive_chunk(s.ctl + us)) return;
  gateup_reduce(p, s, un, pb);
  free_slot(s.ctl + us, s.ctl + kMaxUS + us, it.u + p.n_us);
}

template <int NT, int RG>
__device__ void down_item(const DecParams& p, const Shared& s, const Plan& pl, const Item& it, const Unit& un, int hs,
                          uint8_t* ring, int& slot, Cursor& cu, uint64_t pol, int w, volatile int* abort) {
  const int lane = threadIdx.x & 31, g = lane >> 2, c = lane & 3;
  float acc[NT][2];
#pragma unroll
  for (int nt = 0; nt < NT; ++nt) acc[nt][0] = acc[nt][1] = 0.f;
  // two groups (four tiles) per round where the item has them, as in gate/up
  for (int kt = it.k0; kt < it.k1; kt += 4) {
    uint8_t* sl0 = ring + slot * kGroupBytes;
    const int s1 = slot + 1 == RG ? 0 : slot + 1;
    uint8_t* sl1 = ring + s1 * kGroupBytes;
    if (kt + 2 < it.k1) {
      cp_async_wait<RG - 2>();
      __syncwarp();
      down_tile_smem<NT>(p, s, sl0, kt, un.n, acc);
      down_tile_smem<NT>(p, s, sl0 + kTileBytes, kt + 1, un.n, acc);
      down_tile_smem<NT>(p, s, sl1, kt + 2, un.n, acc);
      if (kt + 3 < it.k1) down_tile_smem<NT>(p, s, sl1 + kTileBytes, kt + 3, un.n, acc);
      __syncwarp();
      issue_group(p, s, pl, w, cu, sl0, pol);
      issue_group(p, s, pl, w, cu, sl1, pol);
      slot = s1 + 1 == RG ? 0 : s1 + 1;
    } else {
      cp_async_wait<RG - 1>();
      __syncwarp();
      down_tile_smem<NT>(p, s, sl0, kt, un.n, acc);
      if (kt + 1 < it.k1) down_tile_smem<NT>(p, s, sl0 + kTileBytes, kt + 1, un.n, acc);
      __syncwarp();
      issue_group(p, s, pl, w, cu, sl0, pol);
      slot = s1;
    }
  }
  const int us = it.u % p.n_us;
  if (!claim_slot(p, s.ctl + 3 * kMaxUS + us, it.u, abort)) return;
  const int hh = min(kHalf, p.tcap);
  float* pb = s.pdn + (size_t)us * kChunks * 16 * hh;
  {
    float* pw = pb + it.c * 16 * hh;  // [16 rows][min(8, tcap) token columns]
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) {
      const int md = 4 * nt + c;
      if (md < un.n) {
        pw[g * hh + md] = acc[nt][0];
        pw[(g + 8) * hh + md] = acc[nt][1];
      }
    }
  }
  if (!arrive_chunk(s.ctl + 2 * kMaxUS + us)) return;
  down_reduce(p, s, un, pb);
  free_slot(s.ctl + 2 * kMaxUS + us, s.ctl + 3 * kMaxUS + us, it.u + p.n_us);
  if (hs == s.misc[4] - 1) {  // the tile's last (slot, half): this warp combines the tile
    __syncwarp();  // the warp's own words are written
    combine_rows(p, s, un.idx, abort);
  }
}

template <int RG, bool kSmall>
__device__ void stream_layer(const DecParams& p, const Shared& s, volatile int* abort) {
  const FwdParams& f = p.f;
  const int w = threadIdx.x >> 5;
  const Plan pl = make_plan(p, s, w);
  const uint64_t pol = evict_first_policy();
  uint8_t* ring = s.ring + (size_t)w * RG * kGroupBytes;
  // The ring first carries the warp's gate/up groups only; its down groups
  // follow once those are consumed, so that while gate/up runs (the critical
  // path up to h) the HBM stream is gate/up weights alone.
  Cursor cu;
  cu.j = 0;
  cu.nitems = pl.nguw;
  cursor_seek(p, s, pl, w, cu);
  for (int i = 0; i < RG; ++i) issue_group(p, s, pl, w, cu, ring + i * kGroupBytes, pol);
  int slot = 0;
  // C: gate/up items
  for (int j = 0; j < pl.nguw; ++j) {
    const Item it = item_of(p, s, pl, w, j);
    const Unit un = gu_unit(p, s, pl.g0 + it.u);
    if (kSmall || un.n <= 8) gateup_item<1, RG>(p, s, pl, it, un, ring, slot, cu, pol, w, abort);
    else gateup_item<2, RG>(p, s, pl, it, un, ring, slot, cu, pol, w, abort);
  }
  // Down groups into the ring (its slots are all consumed; the commits still
  // pending are empty). A warp without gate/up items waits until every warp
  // with some is done, so its down copies do not compete with them.
  if (pl.ndnw > 0) {
    const int with_items = min(kWarps, kChunks * pl.ngu);
    if (pl.nguw == 0 && with_items > 0 && (threadIdx.x & 31) == 0 && ld_acquire_cta_shared(&s.misc[6]) < with_items) {
      const uint64_t t0 = globaltimer();
      while (ld_acquire_cta_shared(&s.misc[6]) < with_items) {
        if (*abort) break;
        if (timed_out(t0, p.wait_ns)) {
          give_up(abort, f.status);
          break;
        }
      }
    }
    __syncwarp();
  }
  if (pl.nguw > 0 && (threadIdx.x & 31) == 0) atomicAdd(&s.misc[6], 1);
  cu.j = pl.nguw;
  cu.nitems = pl.nguw + pl.ndnw;
  cursor_seek(p, s, pl, w, cu);
  for (int i = 0; i < RG; ++i) {
    issue_group(p, s, pl, w, cu, ring + slot * kGroupBytes, pol);
    if (++slot == RG) slot = 0;
  }
  // D: down items, one (slot, half) pair at a time; every warp takes part in
  // every pair's staging barriers, with or without items of that pair
  const int ud = f.d / 16;
  int j = pl.nguw;
  if (pl.ndn > 0) {
    const int hs_first = pl.d0 / ud, hs_last = (pl.d0 + pl.ndn - 1) / ud;
    for (int hs = hs_first; hs <= hs_last; ++hs) {
      // the first barrier ends every read of the shared x / previous h
      named_bar(2, kThreads);
      stage_h(p, s, hs, abort);
      named_bar(2, kThreads);
      for (; j < pl.nguw + pl.ndnw; ++j) {
        const Item it = item_of(p, s, pl, w, j);
        const Unit un = dn_unit(p, s, pl.d0 + it.u);
        if ((pl.d0 + it.u) / ud != hs) break;
        if (kSmall || un.n <= 4) down_item<1, RG>(p, s, pl, it, un, hs, ring, slot, cu, pol, w, abort);
        else down_item<2, RG>(p, s, pl, it, un, hs, ring, slot, cu, pol, w, abort);
      }
    }
  }
  cp_async_wait_all();
}

template <int RG, bool kSmall>
__global__ void __launch_bounds__(kThreads, 1) decode_layer_kernel(DecParams p) {
  extern __shared__ __align__(128) uint8_t sm[];
  Shared s = carve(sm, p);
  volatile int* abort = &s.misc[2];
  const int tid = threadIdx.x;
  if (tid == 0) {
    for (int b = 0; b < kMaxUS; ++b) {
      s.ctl[b] = 0;               // gate/up arrivals
      s.ctl[kMaxUS + b] = b;      // gate/up slot b serves unit b first
      s.ctl[2 * kMaxUS + b] = 0;  // down arrivals
      s.ctl[3 * kMaxUS + b] = b;
    }
    *abort = 0;
    s.misc[6] = 0;
  }
  for (int e = tid; e < p.f.E; e += kThreads) s.cnt[e] = 0;
  stage_router(p, s);
  pdl_wait();  // inputs and workspace are the preceding grid's until here
  if (tid == 0) {
    // launch sequence number: this CTA's word only ever grows, one step per launch,
    // in step with every other CTA's word
    const unsigned seq = p.bar_flags[blockIdx.x] + 1u;
    p.bar_flags[blockIdx.x] = seq;
    s.misc[3] = (int)seq;
  }
  __syncthreads();
  const unsigned seq = (unsigned)s.misc[3];
  stage_x(p, s);
  __syncthreads();
  router(p, s, seq);  // its reads of the bf16 x end before its last barrier (it has none without experts)
  if (!scale_x_beside_topk(p)) {
    scale_x(p, s);
    __syncthreads();
  }
  routing<kSmall>(p, s, seq, abort);
  pdl_launch_dependents();
  stream_layer<RG, kSmall>(p, s, abort);
}

}  // namespace

// Whether the context's calls fit the compact instantiation: E <= 128 (the
// top-k's 4 candidates per lane), at most 4 tokens (one MMA column tile in
// both phases) and at most 32 pairs (the one-warp sort).
bool decode_small(const DecParams& p) {
  return p.f.E <= 128 && p.tcap <= 4 && p.tcap * p.f.k <= 32;
}

// Shared-memory plan of the fused kernel; returns false if it does not fit.
bool decode_plan(DecParams& p, int max_smem, int num_sms) {
  const FwdParams& f = p.f;
  if (f.E > 512 || f.k * kDecodeMaxT > 512) return false;
  auto up = [](size_t v, size_t a) { return (v + a - 1) / a * a; };
  const int hh = std::min(kHalf, p.tcap);
  // f16 row strides 64 bytes past a multiple of 128 (d64, fmax64 are multiples
  // of 64 elements): the 8 rows x 4 16-byte columns of a fragment load hit
  // distinct banks
  p.xstride = f.d64 + 32;
  p.xs_t = p.xstride;  // rows contiguous: K chunks of 128 follow each other
  p.xs_k = 128;
  p.hstride = f.fmax64 + 32;
  size_t off = 4 * kMaxUS * 4;
  off = up(off, 128);
  p.off_x16 = (int)off;
  const size_t xbytes = (size_t)p.tcap * p.xstride * 2;
  const size_t hbytes = (size_t)hh * 2 * p.hstride * 2;
  p.off_hsc = (int)up(off + hbytes, 16);
  const size_t union_end = std::max(off + xbytes, (size_t)p.off_hsc + (size_t)hh * f.hgroups * 4);
  off = up(union_end, 16);
  p.off_xinv = (int)off;
  off = up(off + kDecodeMaxT * 4, 16);
  p.off_red = (int)off;
  off = up(off + (size_t)kWarps * kDecodeMaxT * sizeof(dd), 16);
  const size_t route_bytes = route_region_bytes(f.E, f.k);
  // Each warp's weight ring holds kRing groups: measured on the decode layer,
  // 4 groups per warp (70 KB per SM in flight, about the HBM rate times its
  // latency) beat 8 (25.4 -> 24.2 us per layer), 6, 3 and 2: deeper rings only
  // queue copies that hold up the warp that issues them. The ring region also
  // holds the CTA's router rows during phase A, so it is at least that large.
  const long long router_bytes = (long long)((f.E + 1 + num_sms - 1) / num_sms) * f.d * 4;  // + the gate row
  const size_t ring_bytes = std::max((size_t)kWarps * kRing * kGroupBytes, (size_t)router_bytes);
  for (const int n_us : {kMaxUS, 4, 2}) {
    size_t o = off;
    p.n_us = n_us;
    p.off_pgu = (int)o;
    o = up(o + (size_t)n_us * kChunks * 32 * p.tcap * 4, 16);
    p.off_pdn = (int)o;
    o = up(o + (size_t)n_us * kChunks * 16 * hh * 4, 16);
    p.off_route = (int)o;
    o = up(o + route_bytes, 128);
    p.off_ring = (int)o;
    if ((long long)(o + ring_bytes) <= (long long)max_smem) {
      p.ring_groups = kRing;
      p.smem_bytes = (int)(o + ring_bytes);
      // one CTA per SM: more than half of the shared memory keeps a second CTA out
      if (p.smem_bytes <= max_smem / 2) p.smem_bytes = max_smem / 2 + 128;
      return true;
    }
  }
  return false;
}

cudaError_t configure_decode(int max_smem) {
  cudaError_t e = cudaFuncSetAttribute(decode_layer_kernel<kRing, true>, cudaFuncAttributeMaxDynamicSharedMemorySize, max_smem);
  if (e == cudaSuccess)
    e = cudaFuncSetAttribute(decode_layer_kernel<kRing, false>, cudaFuncAttributeMaxDynamicSharedMemorySize, max_smem);
  return e;
}

int decode_blocks_per_sm(const DecParams& p) {
  int n = 0;
  const cudaError_t e =
      decode_small(p) ? cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, decode_layer_kernel<kRing, true>, kThreads, p.smem_bytes)
                      : cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, decode_layer_kernel<kRing, false>, kThreads, p.smem_bytes);
  return e == cudaSuccess ? n : 0;
}

cudaError_t launch_decode(const DecParams& p, cudaStream_t stream, int num_sms, int max_smem) {
  (void)max_smem;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(num_sms);
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = p.smem_bytes;
  cfg.stream = stream;
  // Programmatic dependent launch: the kernel may be scheduled while the
  // preceding kernel drains; it waits (griddepcontrol.wait) before touching
  // any global memory written by it. The grid is one CTA per SM, each with
  // more than half an SM's shared memory; moe_create checks with the occupancy
  // API that one CTA fits on an SM, so all CTAs of the grid can be resident.
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  if (decode_small(p)) return cudaLaunchKernelEx(&cfg, decode_layer_kernel<kRing, true>, p);
  return cudaLaunchKernelEx(&cfg, decode_layer_kernel<kRing, false>, p);
}

}  // namespace moe
