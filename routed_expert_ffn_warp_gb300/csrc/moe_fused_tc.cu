// The whole MoE layer for T <= 16 tokens in ONE persistent launch on the
// 5th-generation tensor cores: one CTA per SM, 16 warps.
//
//   A  CTA b stages its router rows and x, computes the double-float logits of
//      experts b, b+G, ... and publishes them as launch-tagged words (the
//      routing phases are shared with the mma.sync kernel:
//      moe_fused_route.cuh). It then splits K steps b, b+G, ... of x into two
//      E4M3 planes (the B operand of the gate/up MMAs) in global memory and
//      raises that step's flag to the launch number.
//   B  Every CTA gathers all logits, takes the top k of every token, the
//      softmax gates and the counting sort of the (token, expert) pairs into
//      the slot list (identical results in every CTA).
//   C  Work items, each (unit, K steps) with its MMAs into a TMEM accumulator:
//        gate/up unit (slot, pair p of 128-row M tiles: 64 gate + 64 up rows
//          each), K = d: its epilogue forms h = SiLU(gate) * up of the slot's
//          tokens for f in [128 p, 128 p + 128), splits it into four E4M3
//          planes -- K step p of the slot's down operand -- in global memory
//          and raises that step's flag;
//        down unit (slot, 128-row tile of d), K = the slot's ffn: its B steps
//          wait for the h flags; its epilogue writes the fp32 partial rows,
//          and the CTA finishing a row tile's last slot combines it:
//          y = sum_j g_j part_j (slot order) + shared, one rounding.
//      A CTA takes gate/up units b, b+G, ... and then down units G-1-b,
//      2G-1-b, ...: CTAs without gate/up work start their down weights at
//      once, the rest after their gate/up units. The roles: a weight producer
//      lane (TMA tensor copies that widen the E2M1 codes, plus the scale
//      bytes), an activation producer lane (bulk copies of x or h steps once
//      their flags carry this launch's number), two MMA lanes (M tiles 0 and
//      1 of a unit), each copying its stage's scale factors into tensor memory
//      (tcgen05.cp) ahead of its MMAs, and eight epilogue warps; warps 4-7
//      take part in phases A and B only.
//
// Weights come from the tcgen05 copies of the experts (tc_expert_bytes,
// tc_down_bytes): nothing else is stored. Every wait is bounded; a CTA whose
// wait gives up raises MOE_ERR_TIMEOUT, stops issuing and drains before it
// frees tensor memory. Every reduction runs in a fixed order, so a token's
// output bits do not depend on the other tokens of its call.
//
// The pages: (token, expert) pairs grouped by expert, fused gate/up then down,
// per-token summation over its experts in a fixed order ("NInfer"
// Qwen3.8-Flash-Next notes, MoE execution bullets); the router and top-k step
// that emits each token's expert ids and weights on the GPU ("Neural Server"
// technical page, "How one token and one prompt are processed").
#include <cuda.h>
#include <stdint.h>

#include "../../include/moe.h"
#include "moe_device.cuh"
#include "moe_fused_route.cuh"
#include "moe_internal.h"
#include "moe_tc.cuh"

namespace moe {
namespace {

using namespace dev;

constexpr int kAOp = 128 * kTcStepK;    // one widened E2M1 M tile of a K step: 16 bytes per 16 codes
constexpr int kSfaOff = 2 * kAOp;       // a stage's A scale bytes as stored: 512 per M tile, [lane][4 words]
constexpr int kBOff = 2 * kAOp + 1024;  // a stage's activation slot
constexpr int kAccCols = 64;            // TMEM columns of one accumulator (N <= 64)
// Scale-factor set of stage s at kSfCol0 + 32 s: SFA of M tile 0 / 1 at +0 / +8,
// each MMA lane's own copy of SFB at +16 / +24.
constexpr int kSfCol0 = 256;
constexpr int kMaxStages = 8;
constexpr uint32_t kTmemCols = 512;
constexpr int kProducerWarp = 0, kActWarp = 1, kMmaWarp0 = 2, kEpiWarp0 = 8, kEpiThreads = 256;
constexpr int kHxTok = kDecodeMaxT;     // tokens the gate/up epilogue exchange holds
// K steps (17,408-byte weight blocks, across item boundaries) the producer
// starts towards L2 ahead of its tensor copies: a CTA's few ring stages alone
// keep too few bytes in flight to cover HBM latency, while HBM fills L2 at its
// full rate for every CTA at once. A window, not whole items: whole items of
// the large shapes put most of L2 in flight and evicted their own lines.
// Measured (us per layer, verify | small): 4 steps 73.6 | 53.4, 6 steps
// 74.4 | 54.2, 9 steps 75.5 | 55.2, 12 steps 76.4 | 56.2, 24 steps 81.3 | 56.8.
constexpr int kPfSteps = 4;

__host__ __device__ inline int npad8(int n) { return n <= 8 ? 8 : (n + 7) & ~7; }
__host__ __device__ inline int tc_stage_bytes(int bslot) { return (kBOff + bslot + 1023) / 1024 * 1024; }

// One work item of a CTA: a gate/up or down unit and its K steps.
struct TcItem {
  int down;   // 0: gate/up, 1: down
  int slot;   // slot of the work list
  int e, f;   // expert (E = the shared expert) and its ffn
  int tile;   // tile pair: gate/up M tiles 2p, 2p + 1 (f in [128 p, 128 p + 128)); down rows [256 p, 256 p + 256) of d
  int nt;     // M tiles of the pair holding rows (1 for the last pair of an odd tile count)
  int nks;    // K steps of 128
  int q0, n;  // the slot's rows (pairs in expert order, or the shared expert's tokens)
  int nb;     // B rows: gate/up 2 npad8(T) (x planes of every token), down 4 npad8(n)
};

__device__ __forceinline__ int tc_token_of(const FwdParams& f, const Shared& s, int q) {
  return q < f.P ? s.perm[q] / f.k : q - f.P;
}

// Units of the layer (from the slot list) and this CTA's share of them.
struct TcWork {
  int nr, nsl;      // routed slots, all slots
  int gpF, gpS;     // gate/up units per routed slot and of the shared slot
  int dpp;          // down units per slot (tile pairs of d)
  int ngu, ndn;     // this CTA's gate/up and down items
};

__device__ __forceinline__ TcWork tc_work(const FwdParams& f, const Shared& s) {
  TcWork w;
  w.nr = s.misc[0];
  w.nsl = s.misc[1];
  w.gpF = tc_gu_pairs(f.F);
  w.gpS = f.S > 0 ? tc_gu_pairs(f.S) : 0;
  w.dpp = tc_dn_pairs(f.d);
  const int G = gridDim.x, b = blockIdx.x;
  const int nug = w.nr * w.gpF + (w.nsl > w.nr ? w.gpS : 0);
  const int nud = w.nsl * w.dpp;
  const int bd = G - 1 - b;
  w.ngu = nug > b ? (nug - b + G - 1) / G : 0;
  w.ndn = nud > bd ? (nud - bd + G - 1) / G : 0;
  return w;
}

__device__ __forceinline__ TcItem tc_item(const FwdParams& f, const Shared& s, const TcWork& w, int i) {
  const int G = gridDim.x, b = blockIdx.x;
  TcItem it;
  if (i < w.ngu) {
    const int u = b + i * G;
    it.down = 0;
    if (u < w.nr * w.gpF) {
      it.slot = u / w.gpF;
      it.tile = u - it.slot * w.gpF;
    } else {
      it.slot = w.nr;
      it.tile = u - w.nr * w.gpF;
    }
  } else {
    const int v = (G - 1 - b) + (i - w.ngu) * G;
    it.down = 1;
    it.slot = v / w.dpp;
    it.tile = v - it.slot * w.dpp;
  }
  it.e = s.slot_e[it.slot];
  it.f = it.e == f.E ? f.S : f.F;
  it.q0 = s.slot_q0[it.slot];
  it.n = s.slot_n[it.slot];
  if (it.down) {
    it.nt = min(2, tc_dtiles(f.d) - 2 * it.tile);
    it.nks = tc_ksteps(it.f);
    it.nb = 4 * npad8(it.n);
  } else {
    it.nt = min(2, tc_msteps(it.f) - 2 * it.tile);
    it.nks = tc_ksteps(f.d);
    it.nb = 2 * npad8(f.T);
  }
  return it;
}

// Byte offset of B row n, element k (0..127) of a K step in the MMA's K-major
// core-matrix order (8 rows x 16 bytes per core matrix, LBO 128, SBO 1024).
__device__ __forceinline__ int bop_off(int n, int k) { return ((n >> 3) * 8 + (k >> 4)) * 128 + (n & 7) * 16 + (k & 15); }
// Byte offset, behind N = nb rows, of the E8M0 scale of B row n and K block kb:
// one 512-byte block of words [lane l][r] for rows 32 r + l (nb <= 128).
__device__ __forceinline__ int bsf_off(int nb, int n, int kb) { return nb * 128 + 16 * (n & 31) + 4 * (n >> 5) + kb; }

// Bounded poll (limit ns) by a whole warp of n launch-tagged flags (acquire):
// every flag in one round of loads (lane l takes flags l, l + 32, ...), so an
// item pays one round trip for all of its K steps, not one per step. False if
// it gave up. Every lane returns the same verdict.
__device__ bool tc_poll_flags_warp(const unsigned* flags, int n, unsigned want, long long limit, const DecParams& p,
                                   volatile int* abort) {
  const int lane = threadIdx.x & 31;
  const uint64_t t0 = globaltimer();
  while (true) {
    bool mine = true;
    for (int k = lane; k < n; k += 32) mine = (ld_acquire_u(flags + k) == want) && mine;
    if (__all_sync(0xffffffffu, mine)) return true;
    int stop = *abort ? 1 : 0;
    if (!stop && timed_out(t0, limit)) {
      if (lane == 0) give_up(abort, p.f.status);
      stop = 1;
    }
    if (__any_sync(0xffffffffu, stop)) return false;
    __nanosleep(64);
  }
}

// Phase A tail: K steps G-1-blockIdx.x, + G, ... of x as two E4M3 planes
// with E8M0 scales per 32-element block (x = 2^sh hi + 2^sl lo), rows n =
// plane * npad + t for every token (padding tokens and elements past d are
// zero), in the MMA's operand order, then the scale block; each step's flag
// is raised to `seq` once its bytes are written. The last CTAs take them:
// they hold the fewest router rows (none when E < G), so the planes are ready
// early and no CTA's routing waits behind them (measured: verify 77.1 -> 76.4,
// small 59.6 -> 58.2 us per layer).
__device__ void publish_x_planes(const TcLayerParams& P, const Shared& s, unsigned seq) {
  const DecParams& p = P.d;
  const FwdParams& f = p.f;
  const int nks = tc_ksteps(f.d), npad = npad8(f.T), nb = 2 * npad;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint16_t* xs = reinterpret_cast<const uint16_t*>(s.x16);
  for (int ks = gridDim.x - 1 - blockIdx.x; ks < nks; ks += gridDim.x) {
    uint8_t* dst = P.xplane + (size_t)ks * P.xp_step;
    // scale words of the rows past the planes (never read by the MMAs) hold 2^0
    for (int o = threadIdx.x; o < 128; o += kThreads) reinterpret_cast<uint32_t*>(dst + nb * 128)[o] = 0x7F7F7F7Fu;
    __syncthreads();
    for (int item = warp; item < npad * 4; item += kWarps) {  // (token t, 32-element block j)
      const int t = item >> 2, j = item & 3;
      const int kk = 32 * j + lane, k = kTcStepK * ks + kk;
      const float v = (t < f.T && k < f.d) ? __uint_as_float((uint32_t)xs[xs_off(p, t, k)] << 16) : 0.f;
      uint32_t code[2], sc[2];
      tc::split_planes<2>(v, code, sc);
      dst[bop_off(t, kk)] = (uint8_t)code[0];
      dst[bop_off(npad + t, kk)] = (uint8_t)code[1];
      if (lane < 2) dst[bsf_off(nb, lane * npad + t, j)] = (uint8_t)(lane == 0 ? sc[0] : sc[1]);
    }
    __threadfence();
    fence_proxy_async_global();
    __syncthreads();
    if (threadIdx.x == 0) st_release_u(P.xflag + ks, seq);
  }
}

// Phase B without the mma.sync kernel's x scaling and down halves.
__device__ void tc_routing(const DecParams& p, const Shared& s, unsigned seq, volatile int* abort) {
  const int warp = threadIdx.x >> 5;
  if (warp < p.f.T) {
    if (p.f.E <= 128) topk_token<4>(p, s, warp, seq, abort);
    else if (p.f.E <= 256) topk_token<8>(p, s, warp, seq, abort);
    else topk_token<16>(p, s, warp, seq, abort);
  }
  __syncthreads();
  if (p.f.P > 32) {
    bucket_large(p, s);  // the whole CTA sorts
  } else if (warp == 0) {
    bucket_small<0>(p, s);
  } else if (warp == 1 && blockIdx.x == 0) {
    export_counts_small(p, s);
  }
  __syncthreads();
}

// y rows [256 dp, 256 dp + 256) of every token: sum_j g[t,j] part(pair (t, j)) in
// slot order, then the shared expert, one rounding. The 256 epilogue threads.
__device__ void tc_combine_rows(const FwdParams& f, const Shared& s, int dp, int et) {
  // thread et: row 256 dp + et of every token. The loads of kO tokens x kJ
  // pairs are unconditional (a pair that does not count reads partial row 0
  // and adds nothing), so all of them are in flight together: one L2 round
  // trip per round instead of one per pair and token. Sums in pair order.
  const int row = 256 * dp + et;
  if (row >= f.d) return;
  constexpr int kO = 4, kJ = 4;
  static_assert(kO * kJ <= 64, "pair mask");
  const bool shared = f.S > 0 && f.e_begin == 0;
  for (int t0 = 0; t0 < f.T; t0 += kO) {
    float a[kO];
#pragma unroll
    for (int i = 0; i < kO; ++i) a[i] = 0.f;
    for (int j0 = 0; j0 < f.k; j0 += kJ) {
      float v[kO][kJ];
      unsigned long long ok = 0ull;  // bit i kJ + jj: pair (t0 + i, j0 + jj) counts
#pragma unroll
      for (int i = 0; i < kO; ++i)
#pragma unroll
        for (int jj = 0; jj < kJ; ++jj) {
          const int t = t0 + i, j = j0 + jj, pj = t * f.k + j;
          // this shard's pairs only (all of them without sharding)
          const bool c = t < f.T && j < f.k && expert_in_shard(s.ids[pj], f.e_begin, f.e_end);
          ok |= (c ? 1ull : 0ull) << (i * kJ + jj);
          v[i][jj] = __ldcg(f.part + (size_t)(c ? s.inv[pj] : 0) * f.d + row);
        }
#pragma unroll
      for (int i = 0; i < kO; ++i)
#pragma unroll
        for (int jj = 0; jj < kJ; ++jj)
          if ((ok >> (i * kJ + jj)) & 1ull) a[i] = fmaf(s.gates[(t0 + i) * f.k + j0 + jj], v[i][jj], a[i]);
    }
    float sh[kO];
#pragma unroll
    for (int i = 0; i < kO; ++i)
      sh[i] = shared ? __ldcg(f.part + (size_t)(f.P + min(t0 + i, f.T - 1)) * f.d + row) : 0.f;
#pragma unroll
    for (int i = 0; i < kO; ++i) {
      const int t = t0 + i;
      if (t >= f.T) continue;
      float y = a[i];
      if (shared) y += (f.w_sg ? s.sg[t] : 1.f) * sh[i];
      if (f.out_f32) reinterpret_cast<float*>(f.out)[(size_t)t * f.d + row] = y;
      else reinterpret_cast<__nv_bfloat16*>(f.out)[(size_t)t * f.d + row] = __float2bfloat16_rn(y);
    }
  }
}

// Gate/up epilogue of one unit (accumulator buffer acc): per M tile, the gate
// and up sums of every token go through shared memory (hx [4 blocks][token][32
// f]: blocks 0, 1 gate, 2, 3 up), then h = SiLU(gate) * up of the slot's tokens
// is split into four E4M3 planes -- rows plane * npad8(n) + j of the down
// operand, N = 4 npad8(n) rows, not the gate/up item's own B rows -- of the
// slot's h step p (elements 64 (mt % 2) .. + 63), and the step's flag is raised.
__device__ void tc_gateup_epilogue(const TcLayerParams& P, const Shared& s, const TcItem& it, uint32_t trow, int acc,
                                   float* hx, uint64_t* accempty, unsigned seq) {
  const FwdParams& f = P.d.f;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int qd = warp & 3, eg = (warp - kEpiWarp0) >> 2, ew = warp - kEpiWarp0, et = threadIdx.x - kEpiWarp0 * 32;
  // TMEM lane l of a quadrant holds f offset kk within its 32-element block (the pair-tile row order)
  const int kk = 8 * ((lane & 15) >> 2) + 4 * (lane >> 4) + (lane & 3);
  const int npT = npad8(f.T), npd = npad8(it.n), nbd = 4 * npd, nblk = it.f / 32;
  uint8_t* dst = P.hpanel + ((size_t)it.slot * P.hp_ksteps + it.tile) * P.hp_step;
  for (int t = 0; t < it.nt; ++t) {
    const int mt = 2 * it.tile + t;
    named_bar(1, kEpiThreads);  // the previous readers of hx are done
    if (eg == 0) {              // npad8(T) <= 16 columns per plane: one load of each
      float v[16], w[16];
      const uint32_t dcol = trow + kAccCols * (2 * acc + t);
      tc::ld16(dcol, v);
      tc::ld16(dcol + npT, w);
#pragma unroll
      for (int x = 0; x < 16; ++x)
        if (x < npT) hx[(qd * kHxTok + x) * 32 + kk] = v[x] + w[x];
    }
    if (t == it.nt - 1) {
      tc::fence_before();
      mbar_arrive(accempty);  // every accumulator of the unit has been read
    }
    named_bar(1, kEpiThreads);
    const int kh = 64 * (mt & 1);
    for (int w = ew; w < 2 * npd; w += kEpiThreads / 32) {  // (slot row j, f block b)
      const int j = w >> 1, b = w & 1;
      float h = 0.f;
      if (j < it.n && 2 * mt + b < nblk) {
        const int tok = tc_token_of(f, s, it.q0 + j);
        const float g = hx[(b * kHxTok + tok) * 32 + lane], u = hx[((2 + b) * kHxTok + tok) * 32 + lane];
        h = g / (1.f + __expf(-g)) * u;
      }
      uint32_t code[4], sc[4];
      tc::split_planes4_fixed(h, code, sc);
      const int k = kh + 32 * b + lane;
#pragma unroll
      for (int pl = 0; pl < 4; ++pl) dst[bop_off(pl * npd + j, k)] = (uint8_t)code[pl];
      if (lane < 4) {
        const uint32_t sv = lane == 0 ? sc[0] : lane == 1 ? sc[1] : lane == 2 ? sc[2] : sc[3];
        dst[bsf_off(nbd, lane * npd + j, 2 * (mt & 1) + b)] = (uint8_t)sv;
      }
    }
    if ((mt & 1) == 0 && mt + 1 == tc_msteps(it.f)) {
      // an odd M tile count: the step's second half (f past the ffn) is zero with scale 2^0
      for (int o = et; o < nbd * 4; o += kEpiThreads) {
        const int row = o >> 2, kc = 4 + (o & 3);
        *reinterpret_cast<uint4*>(dst + ((row >> 3) * 8 + kc) * 128 + (row & 7) * 16) = make_uint4(0u, 0u, 0u, 0u);
      }
      for (int o = et; o < nbd * 2; o += kEpiThreads) dst[bsf_off(nbd, o >> 1, 2 + (o & 1))] = 127;
    }
  }
  // publish the step: every writer's stores before the flag, for the bulk copies that read them
  __threadfence();
  fence_proxy_async_global();
  named_bar(1, kEpiThreads);
  if (et == 0) st_release_u(P.hflag + (size_t)it.slot * P.hp_ksteps + it.tile, seq);
}

// Down epilogue of one unit (a pair of 128-row tiles of d): the fp32 rows
// part[q0 + j][128 (2 tile + t) + r] (the sum of the four planes' columns),
// then the pair's counter; the CTA that brings it to the slot count combines
// the pair's rows.
__device__ void tc_down_epilogue(const TcLayerParams& P, const Shared& s, const TcItem& it, uint32_t trow, int acc,
                                 uint64_t* accempty, int* dcnt, int* ctl, int nsl) {
  const FwdParams& f = P.d.f;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int qd = warp & 3, eg = (warp - kEpiWarp0) >> 2, et = threadIdx.x - kEpiWarp0 * 32;
  const int npd = it.nb / 4;
  if (eg < it.nt) {  // warps 8-11 read tile 0, warps 12-15 tile 1; npad8(n) <= 16 columns per plane
    const int t = eg, row = 128 * (2 * it.tile + t) + 32 * qd + lane;
    float v[16], w[16];
    const uint32_t dcol = trow + kAccCols * (2 * acc + t);
    tc::ld16(dcol, v);
#pragma unroll
    for (int pl = 1; pl < 4; ++pl) {
      tc::ld16(dcol + pl * npd, w);
#pragma unroll
      for (int x = 0; x < 16; ++x) v[x] += w[x];
    }
    if (row < f.d) {
#pragma unroll
      for (int x = 0; x < 16; ++x)
        if (x < it.n) f.part[(size_t)(it.q0 + x) * f.d + row] = v[x];
    }
  }
  tc::fence_before();
  mbar_arrive(accempty);
  __threadfence();
  named_bar(1, kEpiThreads);
  if (et == 0) ctl[1] = atomicAdd(dcnt + it.tile, 1) == nsl - 1 ? 1 : 0;
  named_bar(1, kEpiThreads);
  if (ctl[1]) {
    __threadfence();
    tc_combine_rows(f, s, it.tile, et);
  }
}

__device__ __forceinline__ Shared tc_carve(uint8_t* sm, const TcLayerParams& P) {
  const DecParams& p = P.d;
  Shared s = {};
  s.ctl = reinterpret_cast<int*>(sm + P.off_ctl);
  s.red = reinterpret_cast<dd*>(sm + p.off_red);
  carve_route(s, sm, p);
  s.ring = sm + P.off_ring;  // phase A: this CTA's router rows, then the staged bf16 x
  s.x16 = reinterpret_cast<__half*>(sm + P.off_ring + P.router_bytes);
  return s;
}

__global__ void __launch_bounds__(kThreads, 1)
    layer_tc_kernel(const TcLayerParams P, const __grid_constant__ CUtensorMap gu2,
                    const __grid_constant__ CUtensorMap dn2) {
  extern __shared__ __align__(1024) uint8_t sm[];
  const DecParams& p = P.d;
  const FwdParams& f = p.f;
  Shared s = tc_carve(sm, P);
  volatile int* abort = &s.misc[2];
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  if (tid == 0) *abort = 0;
  for (int e = tid; e < f.E; e += kThreads) s.cnt[e] = 0;
  stage_router(p, s);
  pdl_wait();  // inputs and workspace are the preceding grid's until here
  if (tid == 0) {
    const unsigned sq = p.bar_flags[blockIdx.x] + 1u;  // this CTA's launch number (in step with every CTA's)
    p.bar_flags[blockIdx.x] = sq;
    s.misc[3] = (int)sq;
  }
  __syncthreads();
  const unsigned seq = (unsigned)s.misc[3];
  const int dtiles = tc_dtiles(f.d);
  // this launch counts in half seq & 1 (zeroed by the previous launch, or at creation) and zeroes the other
  if (blockIdx.x == 0)
    for (int i = tid; i < dtiles; i += kThreads) P.dcnt[(size_t)((seq + 1) & 1) * dtiles + i] = 0;
  int* dcnt = P.dcnt + (size_t)(seq & 1) * dtiles;
  // barriers and tensor memory now (the preceding grid has finished, so no other CTA holds this SM's TMEM)
  const int S = P.stages, sbytes = tc_stage_bytes(P.bslot);
  uint64_t* full = reinterpret_cast<uint64_t*>(sm + P.off_bars);  // both operands of the stage landed
  uint64_t* empty = full + kMaxStages;     // both MMA lanes' reads of the stage completed
  uint64_t* accfull = empty + kMaxStages;  // [2] both MMA lanes' part of the buffer's unit completed
  uint64_t* accempty = accfull + 2;        // [2] the epilogue read the buffer
  uint32_t* tslot = reinterpret_cast<uint32_t*>(accempty + 2);
  int* ctl = s.ctl;
  if (tid == 0) {
    for (int i = 0; i < S; ++i) {
      mbar_init(&full[i], 2);
      mbar_init(&empty[i], 2);
    }
    for (int a = 0; a < 2; ++a) {
      mbar_init(&accfull[a], 2);
      mbar_init(&accempty[a], kEpiThreads);
    }
    fence_mbar_init();
  }
  if (warp == 0) tc::alloc(tslot, kTmemCols);
  stage_x(p, s);
  tc::fence_before();
  __syncthreads();
  tc::fence_after();
  const uint32_t tmem = *tslot;
  router(p, s, seq);
  publish_x_planes(P, s, seq);
  __syncthreads();  // every read of the router rows and the staged x in the ring is done
  // the tensor copies write the first 8 bytes of every 16-byte operand row; the other 8 are zero
  uint8_t* ring = sm + P.off_ring;
  for (int c = tid; c < S * 2 * (kAOp / 16); c += kThreads)
    *reinterpret_cast<uint2*>(ring + (size_t)(c / (2 * (kAOp / 16))) * sbytes + (size_t)(c % (2 * (kAOp / 16))) * 16 +
                              8) = make_uint2(0u, 0u);
  tc::fence_proxy_async();
  tc_routing(p, s, seq, abort);  // ends with a CTA barrier
  pdl_launch_dependents();

  // ---------------------------------------------------------------- expert units on the tensor cores
  const TcWork wk = tc_work(f, s);
  const int nit = wk.ngu + wk.ndn;
  // Every role but the MMA lanes waits with the suspending try_wait: a warp spinning on a barrier takes
  // issue slots from the MMA lane that shares its scheduler.

  if (warp == kProducerWarp) {
    if (lane == 0) {  // weight blocks: a tensor copy of both tiles' codes (widened) and a bulk copy of their scales
      // prefetch cursor: item pi, its K step ps, its first block pbase; pj blocks started so far
      int pi = 0, ps = 0, pn = 0, pj = 0;
      const uint8_t* pbase = nullptr;
      auto prefetch_to = [&](int upto) {
        while (pj < upto && pi < nit) {
          if (ps == 0) {
            const TcItem pt = tc_item(f, s, wk, pi);
            const size_t we = (size_t)weight_index(f, pt.e);
            pbase = (pt.down ? f.tcwd + we * f.tcwd_stride : f.tcw + we * f.tcw_stride) +
                    (size_t)pt.tile * pt.nks * kTcPairBytes;
            pn = pt.nks;
          }
          prefetch_l2(pbase + (size_t)ps * kTcPairBytes, (uint32_t)kTcPairBytes);
          ++pj;
          if (++ps == pn) {
            ps = 0;
            ++pi;
          }
        }
      };
      int j = 0;
      bool ok = true;
      for (int i = 0; i < nit && ok; ++i) {
        const TcItem it = tc_item(f, s, wk, i);
        const size_t stride = it.down ? f.tcwd_stride : f.tcw_stride;  // a multiple of kTcPairBytes
        const size_t we = (size_t)weight_index(f, it.e);  // the expert's place in this context's copy
        const uint8_t* w0 = (it.down ? f.tcwd : f.tcw) + we * stride + (size_t)it.tile * it.nks * kTcPairBytes;
        const int y0 = (int)(we * (stride / 64) + (size_t)it.tile * it.nks * (kTcPairBytes / 64));
        for (int ks = 0; ks < it.nks; ++ks, ++j) {
          const int st = j % S;
          if (j >= S && !tc::bounded_wait_sleep(&empty[st], (uint32_t)((j / S - 1) & 1), f.status, abort)) {
            ok = false;
            break;
          }
          uint8_t* sb = ring + (size_t)st * sbytes;
          // both tiles' 2 x 8,192 code bytes (counted as read from global memory) + 1,024 scale bytes
          mbar_arrive_expect_tx(&full[st], (uint32_t)kTcPairBytes);
          tc::tma_load_2d(sb, it.down ? &dn2 : &gu2, 0, y0 + ks * (kTcPairBytes / 64), &full[st]);
          bulk_g2s(sb + kSfaOff, w0 + (size_t)ks * kTcPairBytes + 2 * kTcCodeBytes, 1024, &full[st]);
          // the window ahead, at most two blocks per step so the first copies are not held back
          prefetch_to(min(j + 1 + kPfSteps, pj + 2));
        }
      }
    }
  } else if (warp == kActWarp) {
    // activation steps: x planes (gate/up) or the slot's h planes (down). The whole warp checks that
    // every K step of the item is published, then lane 0 copies them stage by stage.
    int j = 0;
    bool ok = true;
    for (int i = 0; i < nit && ok; ++i) {
      const TcItem it = tc_item(f, s, wk, i);
      const unsigned* flags = it.down ? P.hflag + (size_t)it.slot * P.hp_ksteps : P.xflag;
      // the timeout test makes the h steps wait for a number no launch writes
      const bool test = it.down && p.test_extra > 0;
      if (!tc_poll_flags_warp(flags, it.nks, test ? seq + (unsigned)p.test_extra : seq,
                              test ? p.test_wait_ns : p.wait_ns, p, abort)) {
        ok = false;
        break;
      }
      int okl = 1;
      if (lane == 0) {
        fence_proxy_async_global();  // the producers' generic stores -> these async-proxy reads
        const uint32_t bytes = (uint32_t)(it.nb * 128 + 512);
        for (int ks = 0; ks < it.nks; ++ks) {
          const int jj = j + ks, st = jj % S;
          if (jj >= S && !tc::bounded_wait_sleep(&empty[st], (uint32_t)((jj / S - 1) & 1), f.status, abort)) {
            okl = 0;
            break;
          }
          const uint8_t* src = it.down ? P.hpanel + ((size_t)it.slot * P.hp_ksteps + ks) * P.hp_step
                                       : P.xplane + (size_t)ks * P.xp_step;
          mbar_arrive_expect_tx(&full[st], bytes);
          bulk_g2s(ring + (size_t)st * sbytes + kBOff, src, bytes, &full[st]);
        }
      }
      ok = __shfl_sync(0xffffffffu, okl, 0) != 0;
      j += it.nks;
    }
  } else if (warp >= kMmaWarp0 && warp < kMmaWarp0 + 2) {
    if (lane == 0) {  // MMA lane t: M tile t of every unit, into accumulator buffer i % 2
      // per step: its tile's scale factors and its own copy of the activation's to TMEM (tcgen05.cp),
      // then the four K = 32 MMAs -- all from this thread, so they run in this order
      const int t = warp - kMmaWarp0;
      int j = 0;
      bool ok = true;
      for (int i = 0; i < nit && ok; ++i) {
        const TcItem it = tc_item(f, s, wk, i);
        const int acc = i & 1;
        if (i >= 2 && !tc::bounded_wait(&accempty[acc], (uint32_t)((i / 2 - 1) & 1), f.status, abort)) break;
        tc::fence_after();
        const uint32_t d = tmem + kAccCols * (2 * acc + t);
        uint32_t idesc[4];
#pragma unroll
        for (int kb = 0; kb < 4; ++kb) idesc[kb] = tc::idesc_mxf4_mxf8(128, it.nb, kb, kb);
        for (int ks = 0; ks < it.nks; ++ks, ++j) {
          const int st = j % S;
          // every lane takes part in every step's hand-off, with or without MMAs
          if (!tc::bounded_wait(&full[st], (uint32_t)((j / S) & 1), f.status, abort)) {
            ok = false;
            break;
          }
          tc::fence_after();
          if (t < it.nt) {
            const uint8_t* sb = ring + (size_t)st * sbytes;
            const uint32_t sfa = tmem + kSfCol0 + 32 * st + 8 * t, sfb = tmem + kSfCol0 + 32 * st + 16 + 8 * t;
            tc::cp_32x128b_x4(sfa, tc::smem_desc(sb + kSfaOff + 512 * t, 128, 128));
            tc::cp_32x128b_x4(sfb, tc::smem_desc(sb + kBOff + it.nb * 128, 128, 128));
            const uint64_t ad = tc::smem_desc(sb + (size_t)t * kAOp, 128, 8 * 128);
            const uint64_t bd = tc::smem_desc(sb + kBOff, 128, 8 * 128);
#pragma unroll
            for (int kb = 0; kb < 4; ++kb)  // K block kb starts 2 kb core matrices on (256 bytes, 16 descriptor units)
              tc::mma_mxf4_mxf8(d, ad + 16 * kb, bd + 16 * kb, idesc[kb], sfa, sfb, (ks > 0 || kb > 0) ? 1u : 0u);
          }
          tc::commit(&empty[st]);
        }
        if (!ok) break;
        tc::commit(&accfull[acc]);
      }
    }
  } else if (warp >= kEpiWarp0) {
    const uint32_t trow = tmem + ((uint32_t)((warp & 3) * 32) << 16);
    float* hx = reinterpret_cast<float*>(sm + P.off_hx);
    for (int i = 0; i < nit; ++i) {
      const TcItem it = tc_item(f, s, wk, i);
      const int acc = i & 1;
      const bool okw = tc::bounded_wait_sleep(&accfull[acc], (uint32_t)((i / 2) & 1), f.status, abort);
      // one verdict for all 256 (the abort flag may rise between two threads' reads of it)
      if (named_bar_or(1, kEpiThreads, !okw || *abort)) break;
      tc::fence_after();
      if (!it.down) tc_gateup_epilogue(P, s, it, trow, acc, hx, &accempty[acc], seq);
      else tc_down_epilogue(P, s, it, trow, acc, &accempty[acc], dcnt, ctl, wk.nsl);
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

}  // namespace

// Shared-memory plan of the tcgen05 layer kernel; false if it does not fit.
bool tc_layer_plan(TcLayerParams& P, int max_smem, int num_sms) {
  DecParams& p = P.d;
  const FwdParams& f = p.f;
  if (f.E > 512 || f.k * kDecodeMaxT > 512 || p.tcap > kDecodeMaxT || p.tcap < 1 || num_sms < 1) return false;
  auto up = [](size_t v, size_t a) { return (v + a - 1) / a * a; };
  P.npad = npad8(p.tcap);
  P.bslot = 4 * P.npad * 128 + 512;
  P.xp_step = 2 * P.npad * 128 + 512;
  P.hp_step = P.bslot;
  size_t off = 0;
  P.off_ctl = 0;
  off = 256;
  p.off_red = (int)off;
  off = up(off + (size_t)kWarps * kDecodeMaxT * sizeof(dd), 16);
  p.off_route = (int)off;
  off = up(off + route_region_bytes(f.E, f.k), 16);
  P.off_hx = (int)off;
  off = up(off + (size_t)4 * kHxTok * 32 * 4, 16);
  P.off_bars = (int)off;
  off = up(off + (size_t)(3 * kMaxStages + 4) * 8 + 16, 1024);
  P.off_ring = (int)off;
  const size_t sb = (size_t)tc_stage_bytes(P.bslot);
  if ((size_t)max_smem < off + 2 * sb) return false;
  P.stages = (int)std::min<size_t>(kMaxStages, ((size_t)max_smem - off) / sb);
  // during routing the ring holds this CTA's router rows and the staged x (rows of ksteps(d) * 128 elements)
  P.router_bytes = (int)up((size_t)((f.E + 1 + num_sms - 1) / num_sms) * f.d * 4, 128);  // + the gate row
  p.xs_t = tc_ksteps(f.d) * kTcStepK;
  p.xs_k = kTcStepK;
  if ((size_t)P.router_bytes + (size_t)p.tcap * p.xs_t * 2 > (size_t)P.stages * sb) return false;
  P.smem_bytes = (int)(off + (size_t)P.stages * sb);
  if (P.smem_bytes <= max_smem / 2) P.smem_bytes = max_smem / 2 + 128;  // one CTA per SM
  return P.smem_bytes <= max_smem;
}

cudaError_t configure_tc_layer(int max_smem) {
  return cudaFuncSetAttribute(layer_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, max_smem);
}

int tc_layer_blocks_per_sm(const TcLayerParams& P) {
  int n = 0;
  return cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, layer_tc_kernel, kThreads, P.smem_bytes) == cudaSuccess ? n
                                                                                                                     : 0;
}

cudaError_t launch_tc_layer(const TcLayerParams& P, cudaStream_t stream, int num_sms) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(num_sms);
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = P.smem_bytes;
  cfg.stream = stream;
  // programmatic dependent launch: scheduled while the preceding kernel drains, it waits
  // (griddepcontrol.wait) before touching anything that kernel writes
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, layer_tc_kernel, P, *static_cast<const CUtensorMap*>(P.d.f.tmap_gu),
                            *static_cast<const CUtensorMap*>(P.d.f.tmap_dn));
}

}  // namespace moe
