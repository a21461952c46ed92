// Internal structures shared by the host side (moe_api.cu) and the kernels
// (moe_kernels.cu) of the routed-expert FFN library. Not part of the ABI.
#pragma once
#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

namespace moe {

// ---------------------------------------------------------------- packed weight tiles
//
// Every MXFP4 matrix (R rows x K columns, K along the reduction axis) is stored
// as tiles of 16 rows x 64 columns: 512 code bytes followed by 32 scale bytes
// (kTileBytes = 544, 16-byte aligned). Lane L = 4*g + c of a warp owns code
// bytes [16L, 16L+16) of a tile:
//   [0,4)   row g,   block 0 of the tile, code bytes 4c..4c+3 of that block
//   [4,8)   row g+8, block 0
//   [8,12)  row g,   block 1
//   [12,16) row g+8, block 1
// and the quad of lanes with the same g shares the 4 scale bytes at 512 + 4g:
//   scale(row g, block 0), scale(row g+8, block 0), scale(row g, block 1),
//   scale(row g+8, block 1).
// A "block" is one 32-element scale block (16 code bytes). Columns past K are
// padding: code 0 and scale 127. One warp-wide 16-byte load per lane therefore
// brings exactly the A fragments of four m16n8k16 MMAs (two per block).
//
// Which 16 rows a tile holds:
//   down [d x f]:     tile m holds rows 16m .. 16m+15.
//   gate/up [2f x d]: pair-tile tau holds gate rows S_tau and up rows f + S_tau,
//                     S_tau[r] = 32*(tau/2) + 8*(r/4) + 4*(tau%2) + (r%4),
//                     which is the element set one MMA of the down projection
//                     consumes, so h can be scaled per MMA (see the kernels).
// Expert layout: gate/up tiles ordered [tau][kt][gate, up], then down tiles
// ordered [m][kt].
constexpr int kTileBytes = 544;
constexpr int kTileCodeBytes = 512;

__host__ __device__ inline int k64_tiles(int K) { return (K + 63) / 64; }
__host__ __device__ inline size_t gu_packed_bytes(int d, int f) {
  return (size_t)(f / 16) * (size_t)k64_tiles(d) * 2 * kTileBytes;
}
__host__ __device__ inline size_t dn_packed_bytes(int d, int f) {
  return (size_t)(d / 16) * (size_t)k64_tiles(f) * kTileBytes;
}
__host__ __device__ inline size_t expert_packed_bytes(int d, int f) {
  return gu_packed_bytes(d, f) + dn_packed_bytes(d, f);
}

// Second copy of the gate/up weights for the block-scaled tcgen05 GEMM of the
// general path. M tile a is the 64 gate rows then the 64 up rows of pair
// tiles 4a .. 4a+3 (M row m: tile t = m / 16 -- pair tile 4a + t % 4, gate if
// t < 4 -- and row m % 16 of it); a K step is 128 elements of d. Per expert,
// blocks of kTcPairBytes ordered [tile pair P = a / 2][K step ks], each
//  * the 8,192 code bytes of M tile 2P, then those of M tile 2P + 1, in
//    core-matrix order: the 8 packed bytes (16 codes, low nibble = even
//    element) of M row m and 16-element chunk kc at ((m / 8) * 8 + kc) * 64 +
//    (m % 8) * 8, so that widening every 8 bytes to 16 (what a TMA copy of the
//    "16 x U4, 16-byte aligned" type does) gives the K-major operand layout of
//    the MMA (LBO 128, SBO 1024) -- one tensor copy takes both tiles;
//  * 512 scale bytes of M tile 2P, then 512 of M tile 2P + 1, as 32-bit words
//    [lane l][r]: byte kb of word (l, r) is the scale of M row 32 r + l in K
//    block 4 ks + kb, the order tcgen05.st writes them to tensor memory.
// Rows of missing pair tiles (also the whole second tile of the last pair
// when the tile count is odd) and K past d are code 0 with scale 127.
constexpr int kTcStepK = 128;
constexpr int kTcCodeBytes = 8192;
constexpr int kTcPairBytes = 2 * kTcCodeBytes + 1024;
__host__ __device__ inline int tc_msteps(int f) { return (f / 16 + 3) / 4; }
__host__ __device__ inline int tc_ksteps(int d) { return (d + kTcStepK - 1) / kTcStepK; }
__host__ __device__ inline int tc_dtiles(int d) { return (d + 127) / 128; }
// Units of the tcgen05 GEMMs per (slot, token block): pairs of M tiles.
__host__ __device__ inline int tc_gu_pairs(int f) { return (tc_msteps(f) + 1) / 2; }
__host__ __device__ inline int tc_dn_pairs(int d) { return (tc_dtiles(d) + 1) / 2; }
__host__ __device__ inline size_t tc_expert_bytes(int d, int f) {
  return (size_t)tc_gu_pairs(f) * tc_ksteps(d) * kTcPairBytes;
}
// Activation panels of the tcgen05 gate/up GEMM: per (slot, block of up to 48
// tokens) and K step, the B operand -- N = 2 npad rows, row n = plane * npad
// + m (hi plane rows, then lo plane rows; npad = tokens rounded up to 8, at
// least 8) -- in core-matrix order ((n / 8) * 8 + kc) * 128 + (n % 8) * 16,
// directly followed (at N * 128) by 512 scale bytes as words [lane l][r] for
// B row 32 r + l (127 past the rows), so that one bulk copy takes the step.
constexpr int kTcPanelRows = 96;
constexpr int kTcPanelStep = kTcPanelRows * kTcStepK + 512;
// The down projection on the same GEMM: a weight copy of the down matrices in
// the same block format (M tile a = rows 128a .. 128a+127 of d, K steps of 128
// over f; rows past d are code 0 with scale 127) and per-(slot, token block)
// panels of h as four MXFP8 planes (N = 4 npad rows, row n = plane * npad + m,
// up to 192 rows; then, at N * 128, scales as two 512-byte blocks of words
// [lane l][r % 4] for B row 32 r + l, block r / 4), written by the gate/up
// GEMM's epilogue.
constexpr int kTcPanelRowsD = 192;
constexpr int kTcPanelStepD = kTcPanelRowsD * kTcStepK + 1024;
__host__ __device__ inline size_t tc_down_bytes(int d, int f) {
  return (size_t)tc_dn_pairs(d) * tc_ksteps(f) * kTcPairBytes;
}

// ---------------------------------------------------------------- affine group-64 experts
//
// Second weight format: w = scale * q + bias with q an unsigned `bits`-bit code
// and one bf16 scale and one bf16 bias per 64 consecutive weights along the
// reduction axis. Canonical layout per expert (what the load call takes): the
// codes of the gate/up rows [2f][d] then of the down rows [d][f], each row one
// little-endian bit stream (element c at bits [bits c, bits c + bits)); then
// the scales of gate/up [2f][d/64] and of down [d][f/64]; then the biases in
// the same order. The library repacks every expert into tiles of 16 rows x 64
// columns (one group of each row), aff_tile_bytes(bits) bytes:
//  * 128 bits code bytes. Lane L = 4 g + c of a warp owns the `bits` 32-bit
//    words at byte 4 bits L. They carry the lane's 16 code pairs p = 4 kb + r
//    of the m16n8k16 A fragments (kb: k16 block, r: A register): row
//    g + 8 (r & 1), columns 16 kb + 4 c + 2 (r >> 1) and the column after it.
//    Pair p's first code is field p (bits [bits p, bits p + bits)) of a
//    16 bits-bit "first" stream, its second code field p of a "second" stream;
//    word j holds bits [16 j, 16 j + 16) of the first stream in its low half
//    and the same bits of the second stream in its high half, so a shift and a
//    mask give both codes of an A register at once.
//  * 64 bytes: for row pair (g, g + 8) the 64-bit word at 8 g: bf16 scale of
//    row g | scale of row g + 8 << 16, then bias of row g | bias of row g + 8 << 16.
// Gate/up pair tile tau holds gate rows 16 tau .. 16 tau + 15 and up rows
// f + 16 tau ..; tiles ordered [tau][kt][gate, up], then the down tiles [m][kt]
// (rows 16 m ..). A repacked expert has as many bytes as its canonical form.
__host__ __device__ inline int aff_tile_bytes(int bits) { return 128 * bits + 64; }
__host__ __device__ inline size_t aff_gu_bytes(int d, int f, int bits) {
  return (size_t)(f / 16) * (size_t)(d / 64) * 2 * aff_tile_bytes(bits);
}
__host__ __device__ inline size_t aff_expert_bytes(int d, int f, int bits) {
  return (size_t)3 * (size_t)(f / 16) * (size_t)(d / 64) * aff_tile_bytes(bits);
}
// Rows (pairs) per work unit of the affine GEMMs; a gate/up unit = (slot, one
// 16-row pair tile, block of up to kAffRows rows of the slot).
constexpr int kAffRows = 16;
// Row tiles per down work unit of the affine GEMMs: unit = (slot, kAffDnTiles
// 16-row tiles of d, block of rows).
constexpr int kAffDnTiles = 4;

// ---------------------------------------------------------------- forward parameters

struct FwdParams;
// Expert e of the routing (E = the shared expert) -> its index in the
// context's weight copies, which hold experts e_begin .. e_end - 1 and then the
// shared expert.
__host__ __device__ inline bool expert_in_shard(int e, int e_begin, int e_end) { return e >= e_begin && e < e_end; }

constexpr int kRouterSplits = 8;  // most ranges of d the router's fp32 pass splits into
// Multi-kernel path with T <= kRouteDDMaxT: every logit as a double-float sum
// spread over all SMs (router_dd_kernel), the top k inside the bucketing
// kernel (one warp per token); larger T takes the two-pass fp32 router.
constexpr int kRouteDDMaxT = 32;

struct FwdParams {
  // sizes
  int T, d, F, E, k, S;  // S = shared ffn (0 = none)
  int e_begin, e_end;    // experts this context computes (an expert-parallel shard), [0, E) by default;
                         // the shared expert belongs to the shard with e_begin == 0
  int P;                 // T * k
  int d64, fmax64;       // padded row pitches (elements) of x16 and h planes
  int hgroups;           // fmax64 / 16: h scale groups per pair row
  int out_f32;
  // inputs
  const uint16_t* x;     // bf16 [T][d]
  const float* w_router; // [E][d]
  const float* bias;     // [E] or nullptr
  const float* w_sg;     // [d] shared-expert gate row, or nullptr (shared expert added with weight 1)
  const uint8_t* packed; // packed experts (the affine tiles when aff_bits > 0)
  size_t expert_stride;  // packed bytes per routed expert
  int aff_bits;          // 0: MXFP4 experts; 2..8: affine group-64 experts of that code width
  float* xgsum;          // affine: [t_max][xg_pitch] sum of each 64-element group of x16, times 2^-24 (else null)
  int xg_pitch;
  float* hbsum;          // affine: [Q_max][hgroups] sum of each 16-element group of h (as its f16 planes hold
                         // it) times 2^-24; xgsum holds its sums times 2^-24 too
  const void* zeros;     // affine: a zero row (4 max(d64, fmax64) bytes) for absent activation rows
  // workspace
  uint16_t* x16;         // f16 [t_max][d64], x * 2^sigma_t
  float* xinv;           // [t_max]: 2^-sigma_t
  int tc_gateup;         // gate/up on the tcgen05 block-scaled GEMM (moe_tcgemm.cu)
  const uint8_t* tcw;    // its weight copy (see tc_expert_bytes)
  size_t tcw_stride;     // bytes per routed expert of it
  uint8_t* xpanel;       // its activation panels (kTcPanelStep per K step)
  const uint8_t* tcwd;   // the down matrices' copy for the same GEMM (see tc_down_bytes)
  size_t tcwd_stride;    // bytes per routed expert of it
  uint8_t* hpanel;       // h panels of the down step (kTcPanelStepD per K step)
  const void* tmap_gu;   // host: CUtensorMap of tcw (see encode_tc_weight_map)
  const void* tmap_dn;   // host: CUtensorMap of tcwd
  const void* tmap_gu3;  // host: 3-D CUtensorMap of tcw whose box is one tile-pair block (codes + scales)
  const void* tmap_dn3;  // host: the same over tcwd
  int32_t* panel_prefix; // [E+2] first panel of each slot
  uint8_t* xq;           // E4M3 [t_max][2 planes][d64]: x = 2^sh hi + 2^sl lo per 32-element block
  uint8_t* xqs;          // E8M0 [t_max][2][xq_spitch]: the planes' block scales
  int xq_spitch;         // scale bytes per plane row (a multiple of 4)
  float* logit_hi;       // [t_max][E]: exported logits; the first of kRouterSplits planes lstride floats apart
  float* logit_lo;       // = logit_hi + lstride
  size_t lstride;        // t_max * E
  int rsplit;            // ranges of d in the router's fp32 pass (set by the launcher)
  int rsplit_max;        // most ranges the workspace holds planes for (0: kRouterSplits)
  float* xsq;            // [kRouterSplits][t_max]: sums of squares of x_t per range (lstride / E apart)
  float* wsq;            // [kRouterSplits][E]: sums of squares of W_r[e] per range
  int32_t* ids;          // [t_max][k]
  float* gates;          // [t_max][k]
  int32_t* counts;       // [E]
  int32_t* offsets;      // [E+1]
  int32_t* perm;         // [P_max]
  int32_t* inv;          // [P_max]
  // work list (one slot per expert that received pairs, then the shared expert)
  int32_t* n_slots;      // [1]
  int32_t* slot_expert;  // [E+1]  (E = shared)
  int32_t* slot_q0;      // [E+1]  first h/part row of the slot
  int32_t* slot_n;       // [E+1]  rows (pairs) in the slot
  int32_t* gu_prefix;    // [E+2]  prefix of gate/up units (f/16 per slot)
  int32_t* dn_prefix;    // [E+2]  prefix of down units (d/16 per slot)
  uint16_t* hbuf;        // f16 [Q_max][2][fmax64]: hi and lo planes of h * 2^sigma
  float* hscale;         // [Q_max][hgroups]: 2^-sigma per 16-element group
  float* part;           // [Q_max][d]: W_down h of every row q
  void* out;             // [T][d] bf16 or fp32
  int* status;           // device status word
};

// Fused single-kernel decode path (moe_decode.cu), used for T <= kDecodeMaxT.
constexpr int kDecodeMaxT = 16;
// Copies of every published router logit word of the fused path (readers spread over them).
constexpr int kLogitWordCopies = 8;
// Contexts whose t_max * k exceeds this many (token, expert) pairs keep the
// tcgen05 weight layout (fused tcgen05 kernel for T <= 16, tcgen05 GEMMs
// above); smaller ones keep the packed tiles of the fused mma.sync kernel.
// Measured on the decode shapes: T=1, k=4 runs faster on the mma.sync kernel
// (the tcgen05 MMA of a K=32 block costs about 100 cycles whatever N, which
// caps a CTA near 40 GB/s of weights); T=8, k=8 and T=16, k=4 run faster on
// the tcgen05 paths.
constexpr int kFusedMaxPairs = 16;
struct DecParams {
  FwdParams f;
  unsigned long long* hwords;   // [Qd][fmax64] h as (f16 hi | f16 lo << 16) << 32 | launch sequence
  unsigned long long* hswords;  // [Qd][hgroups] its per-16 scales: (fp32 bits << 32) | launch sequence
  unsigned long long* pwords;   // [Qd][d] partial down rows: (fp32 bits << 32) | launch sequence
  unsigned* bar_flags;  // [grid] per-CTA launch sequence numbers (each only grows)
  unsigned long long* lwords;  // [kLogitWordCopies][tcap][E][2] published logits: (fp32 bits << 32) | sequence
  int tcap;             // tokens the x16 shared area holds (min(t_max, kDecodeMaxT))
  int ring_groups;      // 1,088-byte slots of each warp's weight ring
  int n_us;             // partial-sum unit slots per phase
  int xstride, hstride; // f16 row strides of the shared x and h
  int xs_t, xs_k;       // staged bf16 x: element i of token t at t * xs_t + (i / 128) * xs_k + i % 128
  int off_x16, off_hsc, off_xinv, off_red, off_pgu, off_pdn, off_route, off_ring, smem_bytes;
  long long wait_ns;       // bound of every device-side wait
  int test_extra;          // > 0: the h staging waits for a launch number no launch writes (timeout test)
  long long test_wait_ns;  // bound of that wait
};
// Fused single-launch layer on the 5th-generation tensor cores
// (moe_fused_tc.cu), used for T <= kDecodeMaxT when the context holds the
// tcgen05 weight copies. Routing as in the mma.sync kernel (the DecParams
// part); gate/up and down as block-scaled tcgen05 MMAs of TMA-loaded weight
// tiles by MXFP8 activation steps that other CTAs of the same launch publish
// in global memory behind launch-tagged flags.
struct TcLayerParams {
  DecParams d;          // routing: sizes, inputs, workspace, logit words, launch numbers, smem of the routing arrays
  int npad;             // rows per activation plane the context plans for (tcap rounded up to 8, at least 8)
  int stages;           // pipeline stages of the ring
  int bslot;            // bytes of a stage's activation slot: 4 npad rows * 128 + 512
  int off_ctl, off_hx, off_bars, off_ring, smem_bytes;
  int router_bytes;     // this CTA's router rows staged at the start of the ring
  uint8_t* xplane;      // [ksteps(d)][xp_step]: x as two E4M3 planes per K step (rows, then 512 scale bytes)
  int xp_step;          // bytes per x plane step: 2 npad * 128 + 512
  unsigned* xflag;      // [ksteps(d)]: launch number of the published x step
  uint8_t* hpanel;      // [max_slots][hp_ksteps][hp_step]: h of a slot as four E4M3 planes per K step
  int hp_step;          // bytes per h step: 4 npad * 128 + 512
  int hp_ksteps;        // K steps per slot: ksteps(max(ffn, shared ffn))
  int max_slots;        // slots a forward can have: min(E, tcap * k) + (shared expert)
  unsigned* hflag;      // [max_slots][hp_ksteps]: launch number of the published h step
  int* dcnt;            // [2][dtiles(d)]: down units finished per 128-row tile; launches alternate halves
};
bool tc_layer_plan(TcLayerParams& p, int max_smem, int num_sms);
cudaError_t launch_tc_layer(const TcLayerParams& p, cudaStream_t stream, int num_sms);
cudaError_t configure_tc_layer(int max_smem);
int tc_layer_blocks_per_sm(const TcLayerParams& p);

bool decode_plan(DecParams& p, int max_smem, int num_sms);
cudaError_t launch_decode(const DecParams& p, cudaStream_t stream, int num_sms, int max_smem);
// CTAs of the fused kernel (with the shared memory of plan p) that fit on one
// SM of the current device; the fused path needs at least one.
int decode_blocks_per_sm(const DecParams& p);

// Per-device kernel attributes (the dynamic shared-memory limits of the large
// kernels). cudaFuncSetAttribute applies to the current device only, so
// moe_create calls these with its device current, for every context.
cudaError_t configure_decode(int max_smem);
cudaError_t configure_tcgemm(int max_smem);
cudaError_t configure_gemm();
cudaError_t configure_kernels();  // the bucketing kernel's shared-memory limit (moe_kernels.cu)

// Expert GEMMs of the general path (moe_gemm.cu). Work units: (slot, group of
// kGemmTiles 16-row weight tiles, block of up to kGemmRows rows of the slot);
// gu_prefix / dn_prefix hold the running unit counts per slot.
constexpr int kGemmRows = 48;
constexpr int kGemmTiles = 12;
cudaError_t launch_gemm_down(const FwdParams& p, cudaStream_t stream, int num_sms);
// Gate/up of the general path on tcgen05 block-scaled MMAs (moe_tcgemm.cu):
// units (slot, 4 pair tiles, block of up to kTcGemmRows tokens); gu_prefix
// holds their running counts per slot.
constexpr int kTcGemmRows = 48;
cudaError_t launch_gemm_gateup_tc(const FwdParams& p, cudaStream_t stream, int num_sms);
// The activation panels of the tcgen05 gate/up GEMM: x as two MXFP8 planes,
// then one panel per (slot, token block) and K step.
cudaError_t launch_panels_tc(const FwdParams& p, cudaStream_t stream);
cudaError_t launch_gemm_gateup(const FwdParams& p, cudaStream_t stream, int num_sms);
// The same GEMMs for affine group-64 experts (moe_affine.cu): gu_prefix /
// dn_prefix count their units when aff_bits > 0.
cudaError_t configure_affine();
bool affine_bits_supported(int bits);
cudaError_t launch_affine_gateup(const FwdParams& p, cudaStream_t stream, int num_sms);
cudaError_t launch_affine_down(const FwdParams& p, cudaStream_t stream, int num_sms);
// Affine tiles of n_exp experts (ffn f) from their canonical bytes (canon_stride
// apart); a scale or bias that is not finite sets *err_flag.
cudaError_t launch_repack_affine(const uint8_t* canon, int n_exp, int d, int f, int bits, size_t canon_stride,
                                 uint8_t* out, size_t out_stride, int* err_flag, cudaStream_t stream);

// Launchers (moe_kernels.cu). All are asynchronous on `stream`.
// `events` (may be null) receives forward_phases(p) + 1 cudaEvent_t to record
// at the phase boundaries. The register-decode path has 4 phases; the tcgen05
// path 5, so that its two GEMMs are phases of one kernel each.
constexpr int kForwardPhases = 4;
constexpr int kForwardPhasesTc = 5;
extern const char* const kForwardPhaseNames;    // "route,gateup,down,combine"
extern const char* const kForwardPhaseNamesTc;  // "route,panels,gateup,down,combine"
inline int forward_phases(const FwdParams& p) { return p.tc_gateup ? kForwardPhasesTc : kForwardPhases; }
constexpr int kLaunchesPerForward = 7;
constexpr int kLaunchesPerForwardTc = 8;  // no f16 x; + x planes, x panels (tcgen05 GEMMs)
cudaError_t launch_forward(const FwdParams& p, cudaStream_t stream, int num_sms, cudaEvent_t const* events);
__host__ __device__ inline int weight_index(const FwdParams& f, int e) {
  return e == f.E ? f.e_end - f.e_begin : e - f.e_begin;
}
// Routing only (router logits, top-k gates, counting sort) of the general path.
cudaError_t launch_route(const FwdParams& p, cudaStream_t stream);
// Router logits and top-k of the multi-kernel path (moe_kernels.cu).
// with_prep_x: also the f16 x (and affine group sums) for the register-decode / affine GEMMs when T <= 32.
void launch_router(FwdParams p, cudaStream_t stream, bool with_prep_x);
cudaError_t launch_repack(const uint8_t* codes, const uint8_t* scales, int n_exp, int d, int f,
                          size_t canon_code_stride, size_t canon_scale_stride, uint8_t* out, size_t out_stride,
                          int* err_flag, cudaStream_t stream);
// The tcgen05 weight copies of n_exp experts from the canonical layout: gate/up
// (down = false) or down (down = true).
// A scale byte 0xFF (NaN) sets *err_flag.
cudaError_t launch_repack_tc(const uint8_t* codes, const uint8_t* scales, int n_exp, int d, int f,
                             size_t canon_code_stride, size_t canon_scale_stride, uint8_t* out, size_t out_stride,
                             bool down, int* err_flag, cudaStream_t stream);
cudaError_t launch_gemm_down_tc(const FwdParams& p, cudaStream_t stream, int num_sms);
// Dynamic shared memory of the tcgen05 GEMM kernel for E experts.
size_t tc_gemm_smem_bytes(int E, bool down);
// Fills `map` (a 64-byte aligned CUtensorMap) with the tensor map the tcgen05
// kernels load a weight copy of `bytes` bytes at `base` through, with a box of
// box_rows rows of 64 bytes (256: both tiles of a pair's K step; 128: one
// tile); false if the driver refuses it.
bool encode_tc_weight_map(const void* base, size_t bytes, void* map, int box_rows);
// A 3-D tensor map over the same copy whose box is one whole tile-pair block
// (codes and scale bytes of a K step: kTcPairBytes read, twice that written).
bool encode_tc_block_map(const void* base, size_t bytes, void* map);

// Launches a kernel of the forward chain with programmatic stream
// serialization: it may be scheduled once the grid before it has passed its
// own dependency wait. Every such kernel starts with dev::pdl_enter().
template <typename... KArgs, typename... Args>
cudaError_t launch_chained(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t stream,
                           Args&&... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, static_cast<Args&&>(args)...);
}

}  // namespace moe
