// Phases A and B of the fused single-launch layer kernels (the mma.sync
// decode kernel in moe_decode.cu and the tcgen05 kernel in moe_fused_tc.cu),
// shared by both: the double-float router over this CTA's experts with the
// logits published as launch-tagged 64-bit words, the top-k of every token
// from those words (a dataflow exchange: no grid barrier), and the counting
// sort of the (token, expert) pairs into the slot list. Every CTA computes the
// same routing; CTA 0 exports it.
//
// The pages: a router and top-k step yielding the expert ids and weights of
// every token ("Neural Server" technical page, "How one token and one prompt
// are processed"); (token, expert) pairs grouped by expert, weights
// renormalised per token ("NInfer" Qwen3.8-Flash-Next notes, MoE execution).
#pragma once
#include <stdint.h>

#include "../../include/moe.h"
#include "moe_device.cuh"
#include "moe_internal.h"

namespace moe {
namespace {

using namespace dev;

constexpr int kThreads = 512;
constexpr int kWarps = 16;
constexpr int kLogitCopies = kLogitWordCopies;  // CTA b polls copy b % kLogitCopies

struct Shared {
  int* ctl;     // [0, 8) gate/up arrivals, [8, 16) gate/up slot owners, [16, 24) down arrivals, [24, 32) down owners
  __half* x16;  // phase C: [tcap][xstride] f16 x * 2^sigma_t
  __half* hst;  // phase D (same memory): [kHalf][2][hstride] f16 h planes of one (slot, half)
  float* hsc;   //   [kHalf][hgroups] their scales
  float* xinv;  // [16]
  dd* red;      // [12 warps][16 tokens] router partials
  float* pgu;   // [n_us][3 chunks][2][16 rows][tcap] gate/up partial sums
  float* pdn;   // [n_us][3 chunks][16 rows][min(8, tcap)] down partial sums
  int* ids;
  float* gates;
  int* cnt;
  int* offs;
  int* perm;
  int* inv;
  int* slot_e;
  int* slot_n;
  int* slot_q0;
  int* hs_slot;  // (slot, half) list of the down phase
  int* hs_half;
  float* sg;  // [16] shared-expert gate of each token (when the context has a gate row)
  int* misc;  // [0] n_routed, [1] n_slots, [2] abort, [3] launch sequence number,
              // [4] (slot, half) pairs, [5] pairs of routed slots, [6] warps done with their gate/up items
  uint8_t* ring;  // [16 warps][ring_groups][kGroupBytes]
};

// The routing arrays of both kernels at p.off_route (route_region_bytes long):
// ids, gates [16 k], counts, offsets, perm, inv, the slot list, the (slot,
// half) list of the mma.sync kernel's down phase, and the misc words.
__host__ __device__ inline size_t route_region_bytes(int E, int k) {
  const int Pm = kDecodeMaxT * k;
  return (size_t)(4 * Pm + 5 * (E + 1) + 2 * (E + 1 + 64) + 8 + kDecodeMaxT) * 4;
}
__device__ __forceinline__ void carve_route(Shared& s, uint8_t* sm, const DecParams& p) {
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
  s.hs_slot = s.slot_q0 + E + 1;
  s.hs_half = s.hs_slot + E + 1 + 64;
  s.misc = s.hs_half + E + 1 + 64;
  s.sg = reinterpret_cast<float*>(s.misc + 8);
}

// Rows of the router phase: the E expert rows, then the shared-expert gate row
// (when the context has one) as row E, whose dot product with x_t is published
// beside the logits but takes no part in the top k. The logit words have E + 1
// columns per token.
__device__ __forceinline__ int router_rows(const FwdParams& f) { return f.E + (f.w_sg ? 1 : 0); }
__device__ __forceinline__ const float* router_row(const FwdParams& f, int e) {
  return e < f.E ? f.w_router + (size_t)e * f.d : f.w_sg;
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

// ---------------------------------------------------------------- phase A: x, router, x scaling

// Published logit word: (fp32 bits << 32) | launch sequence number.
__device__ __forceinline__ unsigned long long pack_logit(float v, unsigned seq) {
  return ((unsigned long long)__float_as_uint(v) << 32) | seq;
}

// The router rows of this CTA's experts (blockIdx.x, + G, ...) are copied into
// shared memory (the weight ring, idle until phase C) before the kernel waits
// for the preceding grid: the router weights are constant inputs of the layer.
__device__ void stage_router(const DecParams& p, const Shared& s) {
  const int d4 = p.f.d / 4;
  float* wsm = reinterpret_cast<float*>(s.ring);
  int r = 0;
  for (int e = blockIdx.x; e < router_rows(p.f); e += gridDim.x, ++r)
    for (int o = threadIdx.x; o < d4; o += kThreads)
      asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(smem_u32(wsm + (size_t)r * p.f.d + 4 * o)),
                   "l"(router_row(p.f, e) + 4 * o)
                   : "memory");
  asm volatile("cp.async.commit_group;" ::: "memory");
}

// Element i of staged token t: x16[t * xs_t + (i / 128) * xs_k + i % 128] (the
// fused decode kernel keeps rows contiguous, xs_k = 128; the tcgen05 kernel
// groups them by 128-element K step).
__device__ __forceinline__ int xs_off(const DecParams& p, int t, int i) {
  return t * p.xs_t + (i >> 7) * p.xs_k + (i & 127);
}

// x rows (bf16, as stored) into the shared x area with cp.async; all threads.
// The wait also covers the router rows staged before.
__device__ void stage_x(const DecParams& p, const Shared& s) {
  const int d8 = p.f.d / 8;
  for (int o = threadIdx.x; o < p.f.T * d8; o += kThreads) {
    const int t = o / d8, i = o - t * d8;
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(smem_u32(s.x16 + xs_off(p, t, 8 * i))),
                 "l"(p.f.x + (size_t)t * p.f.d + 8 * i)
                 : "memory");
  }
  asm volatile("cp.async.commit_group;" ::: "memory");
  asm volatile("cp.async.wait_all;" ::: "memory");
}

// Router logits from the staged weights and bf16 x. Token t is taken by the
// wpt = 16 / T warps [t wpt, (t+1) wpt), each over an interleaved share of d;
// every lane keeps a double-float sum, then a fixed warp tree and a fixed
// tree over the token's warps.
__device__ void router(const DecParams& p, const Shared& s, unsigned seq) {
  const FwdParams& f = p.f;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int d8 = f.d / 8, T = f.T;
  const int wpt = max(1, kWarps / T), t = warp / wpt, q = warp - t * wpt;
  const float* wsm = reinterpret_cast<const float*>(s.ring);
  int r = 0;
  const int LC = f.E + 1;  // logit word columns
  for (int e = blockIdx.x; e < router_rows(f); e += gridDim.x, ++r) {
    const float* wr = wsm + (size_t)r * f.d;
    if (t < T) {
      dd acc = dd{0.f, 0.f};
      for (int o = q * 32 + lane; o < d8; o += 32 * wpt) {
        const float4 w0 = *reinterpret_cast<const float4*>(wr + 8 * o);
        const float4 w1 = *reinterpret_cast<const float4*>(wr + 8 * o + 4);
        const uint4 xv = *reinterpret_cast<const uint4*>(s.x16 + xs_off(p, t, 8 * o));
        dd_mac(acc, __uint_as_float(xv.x << 16), w0.x);
        dd_mac(acc, __uint_as_float(xv.x & 0xFFFF0000u), w0.y);
        dd_mac(acc, __uint_as_float(xv.y << 16), w0.z);
        dd_mac(acc, __uint_as_float(xv.y & 0xFFFF0000u), w0.w);
        dd_mac(acc, __uint_as_float(xv.z << 16), w1.x);
        dd_mac(acc, __uint_as_float(xv.z & 0xFFFF0000u), w1.y);
        dd_mac(acc, __uint_as_float(xv.w << 16), w1.z);
        dd_mac(acc, __uint_as_float(xv.w & 0xFFFF0000u), w1.w);
      }
      for (int o = 16; o; o >>= 1) acc = dd_add(acc, dd_shfl_xor(acc, o));
      if (lane == 0) s.red[warp] = acc;
    }
    __syncthreads();
    // warp t adds token t's wpt warp partials in a fixed tree, then publishes
    if (warp < T) {
      dd v = lane < wpt ? s.red[warp * wpt + lane] : dd{0.f, 0.f};
      for (int o = 8; o; o >>= 1) v = dd_add(v, dd_shfl_xor(v, o));
      if (lane == 0 && f.bias && e < f.E) v = dd_add(v, dd{f.bias[e], 0.f});
      v.hi = __shfl_sync(0xffffffffu, v.hi, 0);  // lane 0's value in every copy
      v.lo = __shfl_sync(0xffffffffu, v.lo, 0);
      if (lane == 0 && e < f.E) {
        f.logit_hi[(size_t)warp * f.E + e] = v.hi;  // debug export
        f.logit_lo[(size_t)warp * f.E + e] = v.lo;
      }
      // the word carries its own value: no other data is published with it;
      // lane r writes copy r (the readers spread over the copies)
      if (lane < kLogitCopies) {
        unsigned long long* w = p.lwords + ((size_t)lane * p.tcap * LC + (size_t)warp * LC + e) * 2;
        st_relaxed_u64(w, pack_logit(v.hi, seq));
        st_relaxed_u64(w + 1, pack_logit(v.lo, seq));
      }
    }
    __syncthreads();
  }
}

// ---------------------------------------------------------------- phase B: routing (redundant per CTA)

// Top-k of token t by one warp: gather its logits of all E experts from the
// published words (polling until every word carries this launch's number),
// k rounds of a three-key warp reduction (logit hi, logit lo, lowest expert
// index), then the softmax of the k selected logits. NPL = experts per lane.
template <int NPL>
__device__ void topk_token(const DecParams& p, const Shared& s, int t, unsigned seq, volatile int* abort) {
  const FwdParams& f = p.f;
  const int lane = threadIdx.x & 31;
  const int E = f.E, k = f.k;
  const unsigned long long* wt =
      p.lwords + ((size_t)(blockIdx.x % kLogitCopies) * p.tcap * (E + 1) + (size_t)t * (E + 1)) * 2;
  float vh[NPL], vl[NPL];
  unsigned valid = 0;
#pragma unroll
  for (int i = 0; i < NPL; ++i)
    if (lane + 32 * i < E) valid |= 1u << i;
  const uint64_t t0 = globaltimer();
  while (true) {
    // every word of the lane in one round of loads, then one check
    unsigned long long a[NPL], b[NPL];
#pragma unroll
    for (int i = 0; i < NPL; ++i) {
      if ((valid >> i) & 1u) ld_relaxed_u64x2(wt + 2 * (lane + 32 * i), a[i], b[i]);
      else a[i] = b[i] = (unsigned long long)seq;
    }
    bool ready = true;
#pragma unroll
    for (int i = 0; i < NPL; ++i) {
      vh[i] = __uint_as_float((unsigned)(a[i] >> 32));
      vl[i] = __uint_as_float((unsigned)(b[i] >> 32));
      ready = ready && (unsigned)a[i] == seq && (unsigned)b[i] == seq;
    }
    if (__all_sync(0xffffffffu, ready)) break;
    if (*abort || timed_out(t0, p.wait_ns)) {
      if (lane == 0) give_up(abort, f.status);
      break;
    }
  }
  // the shared-expert gate of token t: sigmoid of its published dot product (word column E)
  if (f.w_sg && lane == 0) {
    unsigned long long a, b;
    ld_relaxed_u64x2(wt + 2 * E, a, b);
    while (((unsigned)a != seq || (unsigned)b != seq) && !*abort) {
      if (timed_out(t0, p.wait_ns)) {
        give_up(abort, f.status);
        break;
      }
      ld_relaxed_u64x2(wt + 2 * E, a, b);
    }
    const float z = __uint_as_float((unsigned)(a >> 32)) + __uint_as_float((unsigned)(b >> 32));
    s.sg[t] = 1.f / (1.f + expf(-z));
  }
  // keys of the lane's candidates; taken and absent ones are (0, 0)
  unsigned kh[NPL], kl[NPL];
#pragma unroll
  for (int i = 0; i < NPL; ++i) {
    kh[i] = ((valid >> i) & 1u) ? fkey(vh[i]) : 0u;
    kl[i] = ((valid >> i) & 1u) ? fkey(vl[i]) : 0u;
  }
  int sel_id = 0;
  float sel_h = 0.f, sel_l = 0.f;
  for (int j = 0; j < k; ++j) {
    unsigned bh = 0, bl = 0;
    int bi = 0x7fffffff;
#pragma unroll
    for (int i = 0; i < NPL; ++i) lane_best_dd(kh[i], kl[i], lane + 32 * i, bh, bl, bi);
    unsigned mh, ml;
    const int mi = warp_best_dd(bh, bl, bi, mh, ml);
#pragma unroll
    for (int i = 0; i < NPL; ++i) {  // the owner retires the winner
      const bool won = lane + 32 * i == mi;
      kh[i] = won ? 0u : kh[i];
      kl[i] = won ? 0u : kl[i];
    }
    sel_id = lane == j ? mi : sel_id;
    sel_h = lane == j ? unkey(mh) : sel_h;
    sel_l = lane == j ? unkey(ml) : sel_l;
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

// Counting sort of P <= 32 pairs by expert with one warp. Lane q reads every
// pair's expert (broadcast shared-memory loads) and counts for its own pair q
// the pairs of smaller experts (the first sorted position of its expert), of
// its expert, and before it in the stable order (its sorted position); two
// ballots mark the first pair of every expert of the shard (and those with
// more than HALF pairs), and one more pass counts the slots below each: no
// shuffles and no branches in the loops. With HALF > 0 it also lists the
// (slot, half) pairs of the mma.sync kernel's down phase: a slot with more than
// HALF tokens has two, tokens [0, HALF) and [HALF, n).
template <int HALF>
__device__ void bucket_small(const DecParams& p, const Shared& s) {
  const FwdParams& f = p.f;
  const int lane = threadIdx.x & 31;
  const int P = f.P, E = f.E, T = f.T;
  const bool act = lane < P;
  const int e = act ? s.ids[lane] : 0x7fffffff;
  int below = 0, same = 0, rank = 0;
  for (int j = 0; j < P; ++j) {
    const int ej = s.ids[j];
    below += ej < e;
    same += ej == e;
    rank += (ej < e) || (ej == e && j < lane);
  }
  const bool in = act && rank == below && expert_in_shard(e, f.e_begin, f.e_end);  // first pair of a shard expert
  const unsigned firsts = __ballot_sync(0xffffffffu, in);
  const unsigned bigs = HALF > 0 ? __ballot_sync(0xffffffffu, in && same > HALF) : 0u;
  int slot = 0, big = 0;
  for (int j = 0; j < P; ++j) {
    const int ej = s.ids[j];
    slot += ((firsts >> j) & 1u) && ej < e;
    big += ((bigs >> j) & 1u) && ej < e;
  }
  if (act) {
    s.perm[rank] = lane;
    s.inv[lane] = rank;
    if (blockIdx.x == 0) {
      f.perm[rank] = lane;
      f.inv[lane] = rank;
    }
  }
  if (in) {
    s.slot_e[slot] = e;
    s.slot_q0[slot] = below;
    s.slot_n[slot] = same;
    if (HALF > 0) {
      s.hs_slot[slot + big] = slot;
      s.hs_half[slot + big] = 0;
      if (same > HALF) {
        s.hs_slot[slot + big + 1] = slot;
        s.hs_half[slot + big + 1] = 1;
      }
    }
  }
  if (lane == 0) {
    const int ns = __popc(firsts), nh = ns + __popc(bigs);
    s.misc[0] = ns;
    int tot = ns, th = nh;
    if (f.S > 0 && f.e_begin == 0) {  // the shared expert: slot ns, every token
      s.slot_e[ns] = E;
      s.slot_n[ns] = T;
      s.slot_q0[ns] = P;
      ++tot;
      if (HALF > 0) {
        s.hs_slot[th] = ns;
        s.hs_half[th++] = 0;
        if (T > HALF) {
          s.hs_slot[th] = ns;
          s.hs_half[th++] = 1;
        }
      }
    }
    s.misc[1] = tot;
    if (HALF > 0) {
      s.misc[4] = th;
      s.misc[5] = nh;
    }
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
// Counting sort of P > 32 pairs by expert with all kThreads threads of the
// CTA (every thread must call it; ids are in shared memory): per-expert
// counts by shared atomics, one block scan over the experts that yields both
// the offsets and the slot list (count and "has pairs" packed in one word),
// then every pair's stable rank among the earlier pairs of its expert. Three
// CTA barriers instead of a single warp's long dependent chains.
__device__ void bucket_large(const DecParams& p, const Shared& s) {
  const FwdParams& f = p.f;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int E = f.E, T = f.T, P = f.P;
  const bool writer = blockIdx.x == 0;
  int* wsum = s.hs_half;  // [kWarps] scratch (the down halves are built after this)
  for (int q = tid; q < P; q += kThreads) atomicAdd(&s.cnt[s.ids[q]], 1);
  __syncthreads();
  // expert tid: count in the high half, "a slot of this shard" in the low half
  const int c = tid < E ? s.cnt[tid] : 0;
  const int has = (c > 0 && expert_in_shard(tid, f.e_begin, f.e_end)) ? 1 : 0;
  const int v = (c << 16) | has;
  int inc = v;
  for (int o = 1; o < 32; o <<= 1) {
    const int u = __shfl_up_sync(0xffffffffu, inc, o);
    if (lane >= o) inc += u;
  }
  if (lane == 31) wsum[warp] = inc;
  __syncthreads();
  int before = 0;
  for (int w = 0; w < warp; ++w) before += wsum[w];
  const int excl = before + inc - v;
  if (tid < E) {
    const int off = excl >> 16, slot = excl & 0xFFFF;
    s.offs[tid] = off;
    if (has) {
      s.slot_e[slot] = tid;
      s.slot_n[slot] = c;
      s.slot_q0[slot] = off;
    }
    if (writer) {
      f.offsets[tid] = off;
      f.counts[tid] = c;
    }
    if (tid == E - 1) {
      const int total = excl + v, ns = total & 0xFFFF;
      s.offs[E] = total >> 16;
      if (writer) f.offsets[E] = total >> 16;
      s.misc[0] = ns;
      int tot = ns;
      if (f.S > 0 && f.e_begin == 0) {
        s.slot_e[ns] = E;
        s.slot_n[ns] = T;
        s.slot_q0[ns] = P;
        ++tot;
      }
      s.misc[1] = tot;
    }
  }
  __syncthreads();
  // stable ranks: pair q goes after the earlier pairs of its expert
  for (int q = tid; q < P; q += kThreads) {
    const int e = s.ids[q];
    int r = 0;
    for (int q2 = 0; q2 < q; ++q2) r += s.ids[q2] == e;
    const int pos = s.offs[e] + r;
    s.perm[pos] = q;
    s.inv[q] = pos;
    if (writer) {
      f.perm[pos] = q;
      f.inv[q] = pos;
    }
  }
}

}  // namespace
}  // namespace moe
