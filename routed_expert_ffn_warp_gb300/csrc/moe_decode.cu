// Fused decode path: the whole MoE layer for T <= 16 tokens in ONE persistent
// kernel, one CTA per SM (16 warps: 15 consumers in 5 groups of 3, 1 producer).
//
//   A  CTA b computes the double-float router logits of experts b, b+G, ...
//      and publishes each as two 64-bit words (value bits | launch sequence
//      number); meanwhile 4 warps scale x into f16 in shared memory.
//   B  token warps poll the published words of all experts (a dataflow
//      barrier: no grid-wide sync, no atomics), then every CTA redundantly runs
//      top-k + softmax gates, the counting sort of the T*k pairs and the slot
//      list (identical, deterministic results in every CTA).
//   C  gate/up units (slot, 16-row pair tile) are split evenly over the CTAs;
//      each unit goes to a group of 3 consumer warps that split its K tiles in
//      fixed thirds, while the producer warp streams the unit's chunks into a
//      shared-memory ring with cp.async.bulk (TMA) + mbarriers. The group
//      reduces its three partial sums in a fixed order, applies SiLU(gate)*up,
//      and writes h (f16 hi + lo with a power-of-two scale per 16 elements);
//      every finished unit bumps its slot's counter.
//   D  down units (slot, 16 output rows), slot-major: the producer keeps
//      streaming (down tiles arrive while gate/up still runs); a group waits
//      (bounded) for its slot's h, multiplies, writes the partial rows, and the
//      group finishing a row tile's last slot combines it:
//      y = sum_j g_j part_j (slot order j) + shared, one rounding.
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
// CTA per SM and every CTA needs more than half of an SM's shared memory.
#include <stdint.h>

#include <algorithm>

#include "../../include/moe.h"
#include "moe_device.cuh"
#include "moe_internal.h"

namespace moe {
namespace {

using namespace dev;

constexpr int kThreads = 512;
constexpr int kWarps = 16;
constexpr int kGroups = 5;         // consumer groups of 3 warps; a group processes one unit at a time
constexpr int kGroupWarps = 3;
constexpr int kMemBlock = 5;       // member r of a group owns the k tiles kt with (kt / 5) % 3 == r
constexpr int kProd = 15;          // producer warp
constexpr int kRouterWarps = 12;   // warps 0..11 compute logits, 12..15 scale x
constexpr int kStageTiles = 30;    // 544-byte tiles per ring stage: 16,320-byte bulk copies
constexpr int kStageBytes = kStageTiles * kTileBytes;
static_assert(kStageTiles % 2 == 0, "a gate/up tile pair never straddles two stages");

struct Shared {
  uint64_t* full;
  uint64_t* empty;
  int* seq;     // [ns] stage index currently occupying each ring slot
  __half* x16;
  float* xinv;
  dd* red;      // [12 warps][16 tokens] router partials
  float* part;     // [5 groups][2 members][pfloats][32 lanes] group partial sums
  uint64_t* ubar;  // reserved
  int* ids;
  float* gates;
  int* cnt;
  int* offs;
  int* perm;
  int* inv;
  int* slot_e;
  int* slot_n;
  int* slot_q0;
  int* misc;  // [0] n_routed, [1] n_slots, [2] abort, [3] launch sequence number
  uint8_t* ring;
};

__device__ __forceinline__ Shared carve(uint8_t* sm, const DecParams& p) {
  Shared s;
  s.ubar = reinterpret_cast<uint64_t*>(sm);
  s.full = s.ubar + 4;
  s.empty = s.full + p.ns;
  s.seq = reinterpret_cast<int*>(s.empty + p.ns);
  s.x16 = reinterpret_cast<__half*>(sm + p.off_x16);
  s.xinv = reinterpret_cast<float*>(sm + p.off_xinv);
  s.red = reinterpret_cast<dd*>(sm + p.off_pbuf);
  s.part = reinterpret_cast<float*>(sm + p.off_pbuf + kRouterWarps * kDecodeMaxT * sizeof(dd));
  int* r = reinterpret_cast<int*>(sm + p.off_route);
  const int Pm = kDecodeMaxT * p.f.k, E = p.f.E;
  s.ids = r;
  s.gates = reinterpret_cast<float*>(r + Pm);
  s.cnt = r + 2 * Pm;
  s.offs = s.cnt + E;
  s.perm = s.offs + E + 1;
  s.inv = s.perm + Pm;
  s.slot_e = s.inv + Pm;
  s.slot_n = s.slot_e + E + 1;
  s.slot_q0 = s.slot_n + E + 1;
  s.misc = s.slot_q0 + E + 1;
  s.ring = sm + p.off_ring;
  return s;
}

// ---------------------------------------------------------------- bounded waits

__device__ __forceinline__ bool timed_out(uint64_t t0, long long limit) {
  return (long long)(globaltimer() - t0) > limit;
}

__device__ void set_status(int* status, int code) { atomicCAS(status, 0, code); }

__device__ void give_up(volatile int* abort, int* status) {
  *abort = 1;
  set_status(status, MOE_ERR_TIMEOUT);
}

__device__ bool wait_mbar(uint64_t* bar, uint32_t parity, volatile int* abort, long long limit, int* status) {
  if (*abort) return false;
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = globaltimer();
  while (!mbar_try_wait(bar, parity)) {
    if (*abort) return false;
    if (timed_out(t0, limit)) {
      give_up(abort, status);
      return false;
    }
  }
  return true;
}

// A consumer may parity-wait on a ring slot only once the producer has put
// the stage it wants into that slot (a parity test cannot tell phases that are
// two or more apart): spin on the slot's stage stamp, then on the mbarrier.
__device__ bool wait_stage(const DecParams& p, const Shared& s, uint32_t st, volatile int* abort) {
  const uint32_t j = st % p.ns;
  volatile int* sq = s.seq + j;
  if (*sq != (int)st) {
    const uint64_t t0 = globaltimer();
    while (*sq != (int)st) {
      if (*abort) return false;
      if (timed_out(t0, p.wait_ns)) {
        give_up(abort, p.f.status);
        return false;
      }
    }
  }
  return wait_mbar(&s.full[j], (st / p.ns) & 1u, abort, p.wait_ns, p.f.status);
}

__device__ bool wait_counter(const int* ctr, int target, volatile int* abort, long long limit, int* status) {
  if (*abort) return false;
  if (ld_acquire(ctr) >= target) return true;
  const uint64_t t0 = globaltimer();
  while (ld_acquire(ctr) < target) {
    if (*abort) return false;
    if (timed_out(t0, limit)) {
      give_up(abort, status);
      return false;
    }
  }
  return true;
}

// ---------------------------------------------------------------- work units

struct Unit {
  int slot, idx, e, q0, n, f;
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

__device__ __forceinline__ Unit dn_unit(const DecParams& p, const Shared& s, int u) {
  const int ud = p.f.d / 16;
  Unit r;
  r.slot = u / ud;
  r.idx = u - r.slot * ud;
  r.e = s.slot_e[r.slot];
  r.q0 = s.slot_q0[r.slot];
  r.n = s.slot_n[r.slot];
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

// The CTA's weight stream is a sequence of 544-byte tiles: its gate/up units
// (2 * K64(d) tiles each, gate and up of every k tile adjacent), then its down
// units (K64(f) tiles each). Ring stage S holds stream tiles [30 S, 30 S + 30).
__device__ __forceinline__ int dn_tile0(const DecParams& p, const Shared& s, int d0, int i, int n_gu_tiles) {
  const int nrd = s.misc[0] * (p.f.d / 16);
  const int before_r = max(0, min(d0 + i, nrd) - d0);
  const int before_s = i - before_r;
  return n_gu_tiles + before_r * k64_tiles(p.f.F) + before_s * (p.f.S > 0 ? k64_tiles(p.f.S) : 0);
}

// ---------------------------------------------------------------- phase A: router + x scaling

// Published logit word: (fp32 bits << 32) | launch sequence number.
__device__ __forceinline__ unsigned long long pack_logit(float v, unsigned seq) {
  return ((unsigned long long)__float_as_uint(v) << 32) | seq;
}

__device__ void router(const DecParams& p, const Shared& s, unsigned seq) {
  const FwdParams& f = p.f;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int d8 = f.d / 8, T = f.T;
  for (int e = blockIdx.x; e < f.E; e += gridDim.x) {
    dd acc[kDecodeMaxT];
#pragma unroll
    for (int t = 0; t < kDecodeMaxT; ++t) acc[t] = dd{0.f, 0.f};
    const float* wr = f.w_router + (size_t)e * f.d;
    for (int o = tid; o < d8; o += kRouterWarps * 32) {
      const float4 w0 = __ldg(reinterpret_cast<const float4*>(wr) + 2 * o);
      const float4 w1 = __ldg(reinterpret_cast<const float4*>(wr) + 2 * o + 1);
      const float wv[8] = {w0.x, w0.y, w0.z, w0.w, w1.x, w1.y, w1.z, w1.w};
#pragma unroll
      for (int t = 0; t < kDecodeMaxT; ++t) {
        if (t < T) {
          const uint4 xv = __ldg(reinterpret_cast<const uint4*>(f.x + (size_t)t * f.d) + o);
          const uint32_t xw[4] = {xv.x, xv.y, xv.z, xv.w};
#pragma unroll
          for (int j = 0; j < 4; ++j) {
            dd_mac(acc[t], __uint_as_float(xw[j] << 16), wv[2 * j]);
            dd_mac(acc[t], __uint_as_float(xw[j] & 0xFFFF0000u), wv[2 * j + 1]);
          }
        }
      }
    }
#pragma unroll
    for (int t = 0; t < kDecodeMaxT; ++t) {
      if (t < T) {
        dd v = acc[t];
        for (int o = 16; o; o >>= 1) v = dd_add(v, dd_shfl_xor(v, o));
        if (lane == 0) s.red[warp * kDecodeMaxT + t] = v;
      }
    }
    named_bar(1, kRouterWarps * 32);
    if (tid < T) {
      dd v = s.red[tid];
      for (int w2 = 1; w2 < kRouterWarps; ++w2) v = dd_add(v, s.red[w2 * kDecodeMaxT + tid]);
      if (f.bias) v = dd_add(v, dd{f.bias[e], 0.f});
      f.logit_hi[(size_t)tid * f.E + e] = v.hi;  // debug export
      f.logit_lo[(size_t)tid * f.E + e] = v.lo;
      __threadfence();  // orders this CTA's earlier writes (counter zeroing) before the words
      unsigned long long* w = p.lwords + ((size_t)tid * f.E + e) * 2;
      st_relaxed_u64(w, pack_logit(v.hi, seq));
      st_relaxed_u64(w + 1, pack_logit(v.lo, seq));
    }
    named_bar(1, kRouterWarps * 32);
  }
}

// x -> f16 * 2^sigma_t in shared memory, one warp per token (warps 12..15); padding zeroed.
__device__ void scale_x(const DecParams& p, const Shared& s, int w0, int nw) {
  const FwdParams& f = p.f;
  const int lane = threadIdx.x & 31, warp = (threadIdx.x >> 5) - w0;
  const int d8 = f.d / 8;
  for (int t = warp; t < f.T; t += nw) {
    const uint4* xr = reinterpret_cast<const uint4*>(f.x + (size_t)t * f.d);
    float m = 0.f;
    for (int o = lane; o < d8; o += 32) {
      const uint4 v = __ldg(xr + o);
      const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
      for (int j = 0; j < 4; ++j)
        m = fmaxf(m, fmaxf(fabsf(__uint_as_float(w[j] << 16)), fabsf(__uint_as_float(w[j] & 0xFFFF0000u))));
    }
    for (int o = 16; o; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
    const int sg = f16_headroom_exponent(m);
    const float sc = pow2f(sg);
    for (int o = lane; o < d8; o += 32) {
      const uint4 v = __ldg(xr + o);
      const uint32_t w[4] = {v.x, v.y, v.z, v.w};
      uint32_t h[4];
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const __half2 hv =
            __floats2half2_rn(__uint_as_float(w[j] << 16) * sc, __uint_as_float(w[j] & 0xFFFF0000u) * sc);
        h[j] = *reinterpret_cast<const uint32_t*>(&hv);
      }
      *reinterpret_cast<uint4*>(s.x16 + (size_t)t * f.d64 + 8 * o) = make_uint4(h[0], h[1], h[2], h[3]);
    }
    for (int o = d8 + lane; o < f.d64 / 8; o += 32)  // K padding must be finite: zero
      *reinterpret_cast<uint4*>(s.x16 + (size_t)t * f.d64 + 8 * o) = make_uint4(0, 0, 0, 0);
    if (lane == 0) s.xinv[t] = pow2f(-sg);
  }
}

// ---------------------------------------------------------------- phase B: routing (redundant per CTA)

// Order-preserving map of a float to an unsigned key (-0 folded into +0).
__device__ __forceinline__ unsigned fkey(float v) {
  const unsigned u = __float_as_uint(v + 0.f);
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

// Top-k of token t by one warp: gather its logits of all E experts from the
// published words (polling until every word carries this launch's number),
// k rounds of a three-key warp reduction (logit hi, logit lo, lowest expert
// index), then the softmax of the k selected logits. NPL = experts per lane.
template <int NPL>
__device__ void topk_token(const DecParams& p, const Shared& s, int t, unsigned seq, volatile int* abort) {
  const FwdParams& f = p.f;
  const int lane = threadIdx.x & 31;
  const int E = f.E, k = f.k;
  const unsigned long long* wt = p.lwords + (size_t)t * E * 2;
  float vh[NPL], vl[NPL];
  unsigned need = 0;
#pragma unroll
  for (int i = 0; i < NPL; ++i)
    if (lane + 32 * i < E) need |= 1u << i;
  const unsigned valid = need;
  const uint64_t t0 = globaltimer();
  while (true) {
#pragma unroll
    for (int i = 0; i < NPL; ++i) {
      if ((need >> i) & 1u) {
        const int e = lane + 32 * i;
        const unsigned long long a = ld_relaxed_u64(wt + 2 * e), b = ld_relaxed_u64(wt + 2 * e + 1);
        vh[i] = __uint_as_float((unsigned)(a >> 32));
        vl[i] = __uint_as_float((unsigned)(b >> 32));
        if ((unsigned)a == seq && (unsigned)b == seq) need &= ~(1u << i);
      }
    }
    if (!__any_sync(0xffffffffu, need != 0)) break;
    if (*abort || timed_out(t0, p.wait_ns)) {
      if (lane == 0) give_up(abort, f.status);
      break;
    }
  }
  __threadfence();  // acquire: later reads see what the publishers wrote before their words
  unsigned kh[NPL], kl[NPL];
#pragma unroll
  for (int i = 0; i < NPL; ++i) {
    kh[i] = fkey(vh[i]);
    kl[i] = fkey(vl[i]);
  }
  unsigned taken = ~valid;
  int sel_id = 0;
  float sel_h = 0.f, sel_l = 0.f;
  for (int j = 0; j < k; ++j) {
    unsigned bh = 0, bl = 0;
    int bi = 0x7fffffff;
    float fh = 0.f, fl = 0.f;
#pragma unroll
    for (int i = 0; i < NPL; ++i) {
      const bool free_ = !((taken >> i) & 1u);
      if (free_ && (kh[i] > bh || (kh[i] == bh && kl[i] > bl))) {  // equal keys keep the lower index
        bh = kh[i];
        bl = kl[i];
        bi = lane + 32 * i;
        fh = vh[i];
        fl = vl[i];
      }
    }
    const unsigned mh = __reduce_max_sync(0xffffffffu, bh);
    const unsigned ml = __reduce_max_sync(0xffffffffu, bh == mh ? bl : 0u);
    const int mi = (int)__reduce_min_sync(0xffffffffu, (bh == mh && bl == ml) ? (unsigned)bi : 0x7fffffffu);
    const int owner = mi & 31;
    if (owner == lane) taken |= 1u << (mi >> 5);
    const float wh = __shfl_sync(0xffffffffu, fh, owner), wl = __shfl_sync(0xffffffffu, fl, owner);
    if (lane == j) {
      sel_id = mi;
      sel_h = wh;
      sel_l = wl;
    }
  }
  const float top_h = __shfl_sync(0xffffffffu, sel_h, 0), top_l = __shfl_sync(0xffffffffu, sel_l, 0);
  float ex = 0.f;
  if (lane < k) ex = expf((sel_h - top_h) + (sel_l - top_l));
  float sum = ex;
  for (int o = 16; o; o >>= 1) sum += __shfl_xor_sync(0xffffffffu, sum, o);
  if (lane < k) {
    s.ids[t * k + lane] = sel_id;
    s.gates[t * k + lane] = ex / sum;
    if (blockIdx.x == 0) {
      f.ids[t * k + lane] = sel_id;
      f.gates[t * k + lane] = ex / sum;
    }
  }
}

// Counting sort of P <= 32 pairs by expert with one warp: a bitonic sort of
// the keys (expert << 8 | pair) leaves the pairs stably ordered by expert.
__device__ void bucket_small(const DecParams& p, const Shared& s) {
  const FwdParams& f = p.f;
  const int lane = threadIdx.x & 31;
  const int P = f.P, E = f.E, T = f.T;
  unsigned key = lane < P ? ((unsigned)s.ids[lane] << 8) | (unsigned)lane : 0xffffffffu;
  for (int kk = 2; kk <= 32; kk <<= 1)
    for (int jj = kk >> 1; jj > 0; jj >>= 1) {
      const unsigned other = __shfl_xor_sync(0xffffffffu, key, jj);
      const bool up = (lane & kk) == 0, lower = (lane & jj) == 0;
      key = (lower == up) ? min(key, other) : max(key, other);
    }
  const int e = (int)(key >> 8), q = (int)(key & 0xffu);
  const int eprev = __shfl_up_sync(0xffffffffu, e, 1);
  const bool first = lane < P && (lane == 0 || e != eprev);
  const unsigned firsts = __ballot_sync(0xffffffffu, first);
  const int ns = __popc(firsts);
  if (lane < P) {
    s.perm[lane] = q;
    s.inv[q] = lane;
    if (blockIdx.x == 0) f.perm[lane] = q;
  }
  if (first) {
    const int slot = __popc(firsts & ((1u << lane) - 1u));
    const unsigned after = firsts & ~((2u << lane) - 1u);  // next first lane, or P
    const int next = after ? __ffs(after) - 1 : P;
    s.slot_e[slot] = e;
    s.slot_q0[slot] = lane;
    s.slot_n[slot] = next - lane;
  }
  if (lane == 0) {
    s.misc[0] = ns;
    int tot = ns;
    if (f.S > 0) {
      s.slot_e[ns] = E;
      s.slot_n[ns] = T;
      s.slot_q0[ns] = P;
      ++tot;
    }
    s.misc[1] = tot;
  }
}

// Debug export of counts and offsets for the small-P path (CTA 0, a spare warp).
__device__ void export_counts_small(const DecParams& p, const Shared& s) {
  const FwdParams& f = p.f;
  for (int x = (threadIdx.x & 31); x <= f.E; x += 32) {
    int c = 0, o = 0;
    for (int i = 0; i < f.P; ++i) {
      const int ei = s.ids[i];
      c += (ei == x);
      o += (ei < x);
    }
    if (x < f.E) f.counts[x] = c;
    f.offsets[x] = o;
  }
}

// Counting sort for larger P with one warp: histogram, exclusive scan, slots,
// stable ranks within each bucket.
__device__ void bucket_large(const DecParams& p, const Shared& s) {
  const FwdParams& f = p.f;
  const int lane = threadIdx.x & 31;
  const int E = f.E, T = f.T, P = f.P;
  const bool writer = blockIdx.x == 0;
  for (int q = lane; q < P; q += 32) atomicAdd(&s.cnt[s.ids[q]], 1);
  __syncwarp();
  int loc = 0;  // exclusive scan over E <= 512: lane owns experts [16 lane, 16 lane + 16)
  for (int i = 0; i < 16; ++i) {
    const int e = 16 * lane + i;
    if (e < E) loc += s.cnt[e];
  }
  int inc = loc;
  for (int o = 1; o < 32; o <<= 1) {
    const int v = __shfl_up_sync(0xffffffffu, inc, o);
    if (lane >= o) inc += v;
  }
  int run = inc - loc;
  for (int i = 0; i < 16; ++i) {
    const int e = 16 * lane + i;
    if (e < E) {
      s.offs[e] = run;
      run += s.cnt[e];
    }
  }
  if (lane == 31) s.offs[E] = inc;
  __syncwarp();
  int ns = 0;  // slots: the experts that received pairs, in expert order
  for (int e0 = 0; e0 < E; e0 += 32) {
    const int e = e0 + lane;
    const bool has = e < E && s.cnt[e] > 0;
    const unsigned bal = __ballot_sync(0xffffffffu, has);
    if (has) {
      const int pos = ns + __popc(bal & ((1u << lane) - 1u));
      s.slot_e[pos] = e;
      s.slot_n[pos] = s.cnt[e];
      s.slot_q0[pos] = s.offs[e];
    }
    ns += __popc(bal);
  }
  if (lane == 0) {
    s.misc[0] = ns;
    int tot = ns;
    if (f.S > 0) {
      s.slot_e[ns] = E;
      s.slot_n[ns] = T;
      s.slot_q0[ns] = P;
      ++tot;
    }
    s.misc[1] = tot;
  }
  if (writer)
    for (int i = lane; i <= E; i += 32) {
      f.offsets[i] = s.offs[i];
      if (i < E) f.counts[i] = s.cnt[i];
    }
  __syncwarp();
  int* runp = s.cnt;  // the counts are done with; reuse as running offsets
  for (int i = lane; i < E; i += 32) runp[i] = s.offs[i];
  __syncwarp();
  for (int base = 0; base < P; base += 32) {  // stable ranks, pairs in index order
    const int q = base + lane;
    const bool valid = q < P;
    const int e = valid ? s.ids[q] : -1 - lane;
    const unsigned same = __match_any_sync(0xffffffffu, e);
    const int rank = __popc(same & ((1u << lane) - 1u));
    const int before = valid ? runp[e] : 0;
    __syncwarp();
    if (valid && rank == 0) runp[e] = before + __popc(same);
    __syncwarp();
    if (valid) {
      const int pos = before + rank;
      s.perm[pos] = q;
      s.inv[q] = pos;
      if (writer) f.perm[pos] = q;
    }
  }
}

__device__ void routing(const DecParams& p, const Shared& s, unsigned seq, volatile int* abort) {
  const int warp = threadIdx.x >> 5;
  if (warp < p.f.T) {
    if (p.f.E <= 128) topk_token<4>(p, s, warp, seq, abort);
    else if (p.f.E <= 256) topk_token<8>(p, s, warp, seq, abort);
    else topk_token<16>(p, s, warp, seq, abort);
  }
  __syncthreads();
  if (warp == 0) {
    if (p.f.P <= 32) bucket_small(p, s);
    else bucket_large(p, s);
  } else if (warp == 1 && blockIdx.x == 0 && p.f.P <= 32) {
    export_counts_small(p, s);
  }
  __syncthreads();
}

// ---------------------------------------------------------------- phases C + D: producer

// Source address of stream unit `u` of the CTA (gate/up units first).
struct StreamCursor {
  const uint8_t* src;  // next tile of the current unit
  int left;            // tiles left in the current unit
  int u;               // CTA-local unit index across both phases
};

__device__ void producer(const DecParams& p, const Shared& s, volatile int* abort) {
  const FwdParams& f = p.f;
  const int nr = s.misc[0], nsl = s.misc[1];
  const int NUg = nr * (f.F / 16) + (f.S > 0 ? f.S / 16 : 0);
  const int NUd = nsl * (f.d / 16);
  const int K64d = k64_tiles(f.d);
  int g0, g1, d0, d1;
  unit_range(NUg, g0, g1);
  unit_range(NUd, d0, d1);
  const int ngu = g1 - g0, ndn = d1 - d0;
  const int n_tiles = dn_tile0(p, s, d0, ndn, ngu * 2 * K64d);
  auto unit_src = [&](int u, int& tiles) -> const uint8_t* {
    if (u < ngu) {
      const Unit un = gu_unit(p, s, g0 + u);
      tiles = 2 * K64d;
      return f.packed + (size_t)un.e * f.expert_stride + (size_t)un.idx * K64d * 2 * kTileBytes;
    }
    const Unit un = dn_unit(p, s, d0 + (u - ngu));
    const int K64f = k64_tiles(un.f);
    tiles = K64f;
    return f.packed + (size_t)un.e * f.expert_stride + gu_packed_bytes(f.d, un.f) + (size_t)un.idx * K64f * kTileBytes;
  };
  StreamCursor cur;
  cur.u = 0;
  cur.src = (ngu + ndn > 0) ? unit_src(0, cur.left) : nullptr;
  if (ngu + ndn == 0) cur.left = 0;
  const int n_stages = (n_tiles + kStageTiles - 1) / kStageTiles;
  for (int st = 0; st < n_stages; ++st) {
    const uint32_t j = st % p.ns, par = ((st / p.ns) & 1u) ^ 1u;
    wait_mbar(&s.empty[j], par, abort, p.wait_ns, f.status);
    if (*abort) break;
    const int nt = min(kStageTiles, n_tiles - st * kStageTiles);
    *reinterpret_cast<volatile int*>(s.seq + j) = st;
    mbar_arrive_expect_tx(&s.full[j], (uint32_t)nt * kTileBytes);
    uint8_t* dst = s.ring + (size_t)j * kStageBytes;
    const uint8_t* run_src = nullptr;  // pending copy: merged while the source stays contiguous
    uint32_t run_bytes = 0;
    for (int left = nt; left > 0;) {
      if (cur.left == 0) {
        ++cur.u;
        cur.src = unit_src(cur.u, cur.left);
      }
      const int take = min(left, cur.left);
      if (run_src && run_src + run_bytes == cur.src) {
        run_bytes += (uint32_t)take * kTileBytes;
      } else {
        if (run_src) {
          bulk_g2s(dst, run_src, run_bytes, &s.full[j]);
          dst += run_bytes;
        }
        run_src = cur.src;
        run_bytes = (uint32_t)take * kTileBytes;
      }
      cur.src += (size_t)take * kTileBytes;
      cur.left -= take;
      left -= take;
    }
    if (run_src) bulk_g2s(dst, run_src, run_bytes, &s.full[j]);
    if (nt < kStageTiles) mbar_arrive_cnt(&s.empty[j], (uint32_t)(kStageTiles - nt));  // tiles nobody consumes
  }
  // every issued copy lands before the CTA may exit: wait (bounded) on the
  // last phase of each ring slot that was used
  const int used = n_stages < p.ns ? n_stages : p.ns;
  for (int i = 0; i < used; ++i) {
    const int sidx = n_stages - 1 - i;
    const uint32_t j = sidx % p.ns, par = (sidx / p.ns) & 1u;
    const uint64_t t0 = globaltimer();
    while (!mbar_try_wait(&s.full[j], par)) {
      if (timed_out(t0, p.wait_ns)) {
        set_status(f.status, MOE_ERR_TIMEOUT);
        break;
      }
    }
  }
}

// ---------------------------------------------------------------- phases C + D: consumer groups
//
// Group g (3 warps) takes the CTA's units g, g+5, ...; member r of the group
// owns the unit's k tiles kt with (kt / 5) % 3 == r -- a fixed split, so a
// unit's sums do not depend on the batch -- and the three members share every
// ring stage of their unit. After its k tiles each member hands its partial
// sums to member 0, which adds them in the order member 0, 1, 2.

__device__ __forceinline__ int member_first(int r) { return r * kMemBlock; }
__device__ __forceinline__ int member_next(int kt) {
  return ((kt + 1) % kMemBlock) ? kt + 1 : kt + 1 + (kGroupWarps - 1) * kMemBlock;
}

template <int NV>
__device__ __forceinline__ void group_reduce(const DecParams& p, const Shared& s, int grp, int mem, float (&v)[NV]) {
  const int lane = threadIdx.x & 31;
  float* buf = s.part + (size_t)grp * 2 * p.pfloats * 32;
  if (mem > 0) {
#pragma unroll
    for (int i = 0; i < NV; ++i) buf[((size_t)(mem - 1) * p.pfloats + i) * 32 + lane] = v[i];
  }
  named_bar(2 + grp, kGroupWarps * 32);
  if (mem == 0) {
#pragma unroll
    for (int i = 0; i < NV; ++i) v[i] = (v[i] + buf[(size_t)i * 32 + lane]) + buf[((size_t)p.pfloats + i) * 32 + lane];
  }
  named_bar(2 + grp, kGroupWarps * 32);
}

// Release `used` tiles of ring stage `cur` (the empty barrier counts tiles).
__device__ __forceinline__ void release_tiles(const DecParams& p, const Shared& s, int cur, int used) {
  if (cur < 0) return;
  __syncwarp();
  if ((threadIdx.x & 31) == 0) mbar_arrive_cnt(&s.empty[cur % p.ns], (uint32_t)used);
}

template <int NT>
__device__ void gateup_unit(const DecParams& p, const Shared& s, const Unit& un, int t0, int grp, int mem,
                            volatile int* abort) {
  const FwdParams& f = p.f;
  const int lane = threadIdx.x & 31, g = lane >> 2, c = lane & 3;
  const int K64d = k64_tiles(f.d);
  float acc[2 * NT * 4];  // gate then up, n8 tile nt, fragment r
#pragma unroll
  for (int i = 0; i < 2 * NT * 4; ++i) acc[i] = 0.f;
  int tokB[NT];
#pragma unroll
  for (int nt = 0; nt < NT; ++nt) {
    const int m = 8 * nt + g;
    tokB[nt] = (m < un.n) ? token_of(p, s, un.q0 + m) : -1;
  }
  int cur = -1, used = 0;
  bool ok = false;
  for (int kt = member_first(mem); kt < K64d; kt = member_next(kt)) {
    const int tile = t0 + 2 * kt;
    const int st = tile / kStageTiles;
    if (st != cur) {
      release_tiles(p, s, cur, used);
      ok = wait_stage(p, s, (uint32_t)st, abort);
      cur = st;
      used = 0;
    }
    used += 2;
    if (ok) {
      const uint8_t* tg = s.ring + (size_t)(st % p.ns) * kStageBytes + (size_t)(tile % kStageTiles) * kTileBytes;
      const uint8_t* tu = tg + kTileBytes;
      const uint4 qg = *reinterpret_cast<const uint4*>(tg + 16 * lane);
      const uint32_t sgv = *reinterpret_cast<const uint32_t*>(tg + kTileCodeBytes + 4 * g);
      const uint4 qu = *reinterpret_cast<const uint4*>(tu + 16 * lane);
      const uint32_t suv = *reinterpret_cast<const uint32_t*>(tu + kTileCodeBytes + 4 * g);
      uint4 bx[NT][2];
#pragma unroll
      for (int nt = 0; nt < NT; ++nt)
#pragma unroll
        for (int bb = 0; bb < 2; ++bb)
          bx[nt][bb] = tokB[nt] >= 0 ? *reinterpret_cast<const uint4*>(s.x16 + (size_t)tokB[nt] * f.d64 + kt * 64 +
                                                                       bb * 32 + c * 8)
                                     : make_uint4(0, 0, 0, 0);
      float (&ag)[NT][4] = *reinterpret_cast<float(*)[NT][4]>(acc);
      float (&au)[NT][4] = *reinterpret_cast<float(*)[NT][4]>(acc + NT * 4);
      gu_tile<NT>(qg, sgv, bx, ag);
      gu_tile<NT>(qu, suv, bx, au);
    }
  }
  release_tiles(p, s, cur, used);
  group_reduce<2 * NT * 4>(p, s, grp, mem, acc);
  if (mem != 0) return;
  // SwiGLU epilogue (member 0): h for the 16 rows S_tau of this unit and each token column
#pragma unroll
  for (int nt = 0; nt < NT; ++nt) {
    float hv[4];
#pragma unroll
    for (int r = 0; r < 4; ++r) {
      const int m = 8 * nt + 2 * c + (r & 1);
      float h = 0.f;
      if (m < un.n) {
        const float xi = s.xinv[token_of(p, s, un.q0 + m)];
        const float gate = acc[nt * 4 + r] * xi, up = acc[NT * 4 + nt * 4 + r] * xi;
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
      if (m >= un.n) continue;
      const int q = un.q0 + m;
      const int sh = f16_headroom_exponent(col ? mx1 : mx0);
      const float sc = pow2f(sh);
      __half* hi = reinterpret_cast<__half*>(f.hbuf) + (size_t)q * 2 * f.fmax64;
      __half* lo = hi + f.fmax64;
#pragma unroll
      for (int half = 0; half < 2; ++half) {
        const int rr = g + 8 * half;
        const int i = 32 * (un.idx >> 1) + 8 * (rr >> 2) + 4 * (un.idx & 1) + (rr & 3);
        const float v = hv[2 * half + col] * sc;
        const __half vh = __float2half_rn(v);
        hi[i] = vh;
        lo[i] = __float2half_rn(v - __half2float(vh));
      }
      if (g == 0) f.hscale[(size_t)q * f.hgroups + un.idx] = pow2f(-sh);
    }
  }
  __threadfence();
  __syncwarp();
  if (lane == 0) atomicAdd(&p.done[un.slot], 1);
}

template <int NT>
__device__ void down_unit(const DecParams& p, const Shared& s, const Unit& un, int t0, int grp, int mem,
                          volatile int* abort) {
  const FwdParams& f = p.f;
  const int lane = threadIdx.x & 31, g = lane >> 2, c = lane & 3;
  const int K64f = k64_tiles(un.f);
  float acc[2 * NT];
#pragma unroll
  for (int i = 0; i < 2 * NT; ++i) acc[i] = 0.f;
  const uint16_t* hrow[NT];
  const float* srow[NT];
  int qD[NT];
#pragma unroll
  for (int nt = 0; nt < NT; ++nt) {
    const int mb = 4 * nt + (g >> 1), md = 4 * nt + c;
    qD[nt] = (md < un.n) ? un.q0 + md : -1;
    hrow[nt] = (mb < un.n) ? f.hbuf + ((size_t)(un.q0 + mb) * 2 + (g & 1)) * f.fmax64 + c * 8 : nullptr;
    srow[nt] = qD[nt] >= 0 ? f.hscale + (size_t)qD[nt] * f.hgroups : nullptr;
  }
  if (member_first(mem) < K64f) {
    // h of this slot is written by other CTAs: wait (bounded) for all its gate/up units
    if (lane == 0)
      wait_counter(&p.done[un.slot], un.f / 16 + p.test_extra, abort, p.test_extra ? p.test_wait_ns : p.wait_ns,
                   f.status);
    __syncwarp();
  }
  int cur = -1, used = 0;
  bool ok = false;
  // h fragment loads are batched (BATCH k tiles at a time, all loads before the MMAs)
  constexpr int BATCH = NT == 1 ? kMemBlock : 1;
  for (int kb = member_first(mem); kb < K64f; kb = member_next(kb + BATCH - 1)) {
    uint4 bh[BATCH][NT][2];
    float2 sb[BATCH][NT][2];
#pragma unroll
    for (int i = 0; i < BATCH; ++i)
#pragma unroll
      for (int nt = 0; nt < NT; ++nt)
#pragma unroll
        for (int bb = 0; bb < 2; ++bb) {
          const int kt = kb + i;
          const bool in = kt < K64f;
          // plain (L1-cached) loads: h is final once the slot counter was seen
          bh[i][nt][bb] = (in && hrow[nt]) ? *reinterpret_cast<const uint4*>(hrow[nt] + kt * 64 + bb * 32)
                                           : make_uint4(0, 0, 0, 0);
          sb[i][nt][bb] = (in && srow[nt]) ? *reinterpret_cast<const float2*>(srow[nt] + 2 * (2 * kt + bb))
                                           : make_float2(0.f, 0.f);
        }
#pragma unroll
    for (int i = 0; i < BATCH; ++i) {
      const int kt = kb + i;
      if (kt >= K64f) break;
      const int tile = t0 + kt;
      const int st = tile / kStageTiles;
      if (st != cur) {
        release_tiles(p, s, cur, used);
        ok = wait_stage(p, s, (uint32_t)st, abort);
        cur = st;
        used = 0;
      }
      ++used;
      if (ok) {
        const uint8_t* t8 = s.ring + (size_t)(st % p.ns) * kStageBytes + (size_t)(tile % kStageTiles) * kTileBytes;
        const uint4 q = *reinterpret_cast<const uint4*>(t8 + 16 * lane);
        const uint32_t scv = *reinterpret_cast<const uint32_t*>(t8 + kTileCodeBytes + 4 * g);
        float (&a2)[NT][2] = *reinterpret_cast<float(*)[NT][2]>(acc);
        dn_tile<NT>(q, scv, bh[i], sb[i], a2);
      }
    }
  }
  release_tiles(p, s, cur, used);
  group_reduce<2 * NT>(p, s, grp, mem, acc);
  if (mem != 0) return;
#pragma unroll
  for (int nt = 0; nt < NT; ++nt) {
    if (qD[nt] >= 0) {
      float* dst = f.part + (size_t)qD[nt] * f.d + 16 * un.idx;
      dst[g] = acc[2 * nt];
      dst[g + 8] = acc[2 * nt + 1];
    }
  }
  __threadfence();
  __syncwarp();
  int last = 0;
  if (lane == 0) last = atomicAdd(&p.rowcnt[un.idx], 1) == s.misc[1] - 1;
  last = __shfl_sync(0xffffffffu, last, 0);
  if (last) {
    // this group finished the row tile's last slot: combine its 16 rows
    __threadfence();
    const int r0 = 16 * un.idx;
    for (int idx = lane; idx < f.T * 16; idx += 32) {
      const int t = idx >> 4, r = idx & 15;
      float a = 0.f;
      for (int j0 = 0; j0 < f.k; j0 += 4) {  // loads of a group issued together, sums kept in slot order
        float pv[4];
#pragma unroll
        for (int uu = 0; uu < 4; ++uu)
          pv[uu] = (j0 + uu < f.k) ? __ldcg(f.part + (size_t)s.inv[t * f.k + j0 + uu] * f.d + r0 + r) : 0.f;
#pragma unroll
        for (int uu = 0; uu < 4; ++uu)
          if (j0 + uu < f.k) a = fmaf(s.gates[t * f.k + j0 + uu], pv[uu], a);
      }
      if (f.S > 0) a += __ldcg(f.part + (size_t)(f.P + t) * f.d + r0 + r);
      if (f.out_f32) reinterpret_cast<float*>(f.out)[(size_t)t * f.d + r0 + r] = a;
      else reinterpret_cast<__nv_bfloat16*>(f.out)[(size_t)t * f.d + r0 + r] = __float2bfloat16_rn(a);
    }
  }
}

__device__ void consumers(const DecParams& p, const Shared& s, volatile int* abort) {
  const FwdParams& f = p.f;
  const int w = threadIdx.x >> 5;
  const int grp = w / kGroupWarps, mem = w % kGroupWarps;
  const int nr = s.misc[0], nsl = s.misc[1];
  const int NUg = nr * (f.F / 16) + (f.S > 0 ? f.S / 16 : 0);
  const int NUd = nsl * (f.d / 16);
  const int K64d = k64_tiles(f.d);
  int b0, b1;
  unit_range(NUg, b0, b1);
  const int n_gu_tiles = (b1 - b0) * 2 * K64d;
  for (int i = grp; i < b1 - b0; i += kGroups) {
    const Unit un = gu_unit(p, s, b0 + i);
    const int t0 = i * 2 * K64d;
    if (un.n <= 8) gateup_unit<1>(p, s, un, t0, grp, mem, abort);
    else gateup_unit<2>(p, s, un, t0, grp, mem, abort);
  }
  int d0, d1;
  unit_range(NUd, d0, d1);
  for (int i = grp; i < d1 - d0; i += kGroups) {
    const Unit un = dn_unit(p, s, d0 + i);
    const int t0 = dn_tile0(p, s, d0, i, n_gu_tiles);
    if (un.n <= 4) down_unit<1>(p, s, un, t0, grp, mem, abort);
    else if (un.n <= 8) down_unit<2>(p, s, un, t0, grp, mem, abort);
    else if (un.n <= 12) down_unit<3>(p, s, un, t0, grp, mem, abort);
    else down_unit<4>(p, s, un, t0, grp, mem, abort);
  }
}

__global__ void __launch_bounds__(kThreads, 1) decode_layer_kernel(DecParams p) {
  extern __shared__ __align__(128) uint8_t sm[];
  const Shared s = carve(sm, p);
  volatile int* abort = &s.misc[2];
  const int tid = threadIdx.x, warp = tid >> 5;
  if (tid == 0) {
    for (int i = 0; i < p.ns; ++i) {
      mbar_init(&s.full[i], 1);
      mbar_init(&s.empty[i], kStageTiles);
      s.seq[i] = -1;
    }

    fence_mbar_init();
    *abort = 0;
  }
  for (int e = tid; e < p.f.E; e += kThreads) s.cnt[e] = 0;
  pdl_wait();  // inputs and workspace are the preceding grid's until here
  if (tid == 0) {
    // launch sequence number: this CTA's word only ever grows, one step per launch,
    // in step with every other CTA's word
    const unsigned seq = p.bar_flags[blockIdx.x] + 1u;
    p.bar_flags[blockIdx.x] = seq;
    s.misc[3] = (int)seq;
  }
  if (blockIdx.x == 0) {
    for (int i = tid; i <= p.f.E; i += kThreads) p.done[i] = 0;
    for (int i = tid; i < p.f.d / 16; i += kThreads) p.rowcnt[i] = 0;
  }
  __syncthreads();
  const unsigned seq = (unsigned)s.misc[3];
  if (warp < kRouterWarps) router(p, s, seq);
  else scale_x(p, s, kRouterWarps, kWarps - kRouterWarps);
  __syncthreads();
  routing(p, s, seq, abort);
  pdl_launch_dependents();
  if (warp == kProd) {
    if ((tid & 31) == 0) producer(p, s, abort);
  } else {
    consumers(p, s, abort);
  }
}

}  // namespace

// Shared-memory plan of the fused kernel; returns false if it does not fit.
bool decode_plan(DecParams& p, int max_smem) {
  const FwdParams& f = p.f;
  if (f.E > 512 || f.k * kDecodeMaxT > 512) return false;
  p.stage_bytes = kStageBytes;
  auto up = [](size_t v, size_t a) { return (v + a - 1) / a * a; };
  const int Pm = kDecodeMaxT * f.k;
  size_t off = 0;
  const size_t bars_max = 32 + (2 * 8 + 4) * 128;  // 4 unit barriers; up to 128 stages: two mbarriers and a stamp each
  off = bars_max;
  p.off_x16 = (int)off;
  off = up(off + (size_t)p.tcap * f.d64 * 2, 16);
  p.off_xinv = (int)off;
  off = up(off + kDecodeMaxT * 4, 16);
  p.off_pbuf = (int)off;
  p.pfloats = p.tcap <= 8 ? 8 : 16;  // gate/up partials: 8 per n8 token tile (NT = 2 above 8 tokens)
  p.pbuf_depth = 1;
  off = up(off + (size_t)kRouterWarps * kDecodeMaxT * sizeof(dd) + (size_t)kGroups * 2 * p.pfloats * 32 * 4, 16);
  p.off_route = (int)off;
  off = up(off + (size_t)(4 * Pm + 5 * (f.E + 1) + 8) * 4, 128);
  (void)Pm;
  p.off_ring = (int)off;
  const long long room = (long long)max_smem - (long long)off;
  int ns = (int)(room / p.stage_bytes);
  if (ns > 128) ns = 128;
  if (ns < 4) return false;
  p.ns = ns;
  p.smem_bytes = (int)(off + (size_t)ns * p.stage_bytes);
  return true;
}

cudaError_t launch_decode(const DecParams& p, cudaStream_t stream, int num_sms, int max_smem) {
  static int configured = 0;
  if (configured < max_smem) {
    cudaError_t e = cudaFuncSetAttribute(decode_layer_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, max_smem);
    if (e != cudaSuccess) return e;
    configured = max_smem;
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(num_sms);
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = p.smem_bytes;
  cfg.stream = stream;
  // Programmatic dependent launch: the kernel may be scheduled while the
  // preceding kernel drains; it waits (griddepcontrol.wait) before touching
  // any global memory. Co-residency of the grid holds by construction (one
  // CTA per SM, more than half an SM's shared memory each).
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, decode_layer_kernel, p);
}

}  // namespace moe
