/*
 * moe.h -- C ABI of the routed-expert FFN layer for NVIDIA GB300 (sm_103a).
 *
 * One MoE block of a large MoE language model, run entirely on one GPU:
 *
 *   logits  l[t,e] = sum_i W_r[e,i] x[t,i] + b[e]
 *   top-k   ids[t,0..k) = the k largest logits, largest first, ties to the lower e
 *   gates   g[t,j] = softmax of the k selected logits
 *   expert  h = SiLU(W_gate x) * (W_up x),   part = W_down h      (MXFP4 weights)
 *   combine y[t] = sum_j g[t,j] part(t, ids[t,j]) + shared(x_t)  (shared: weight 1)
 *
 * Where the pages define it (page title, section):
 *   "Neural Server" technical page, "How one token and one prompt are
 *     processed": a router + top-k step yields 4 expert ids and 4 weights per
 *     token, then resident experts run as MXFP4 GEMVs on the GPU.
 *   "Neural Server" technical page, "What it runs on and what it runs": 128
 *     experts, four active per token, hidden 2880, 13,219,200 B per expert.
 *   "NInfer" Qwen3.8-Flash-Next notes, MoE execution: (token, expert) pairs are
 *     grouped by expert on the GPU, expert base-pointer tables, fused gate/up
 *     then down, weighted outputs summed in an order-independent way, weights
 *     renormalised per token.
 *   "Running Qwen3.8-Flash-Next on a 32 GB Mac with Transformers",
 *     architecture: one shared expert per layer next to the routed ones.
 * MXFP4 itself follows the OCP Microscaling Formats (MX) v1.0 specification:
 * 4-bit E2M1 codes, one E8M0 scale byte per 32 elements along the reduction
 * axis, value = E2M1(code) * 2^(scale - 127).
 *
 * Canonical weight layout accepted by moe_load_experts (expert-major, one
 * contiguous byte range per expert, as the "NInfer" notes describe banks):
 *   codes : expert j starts at j * (3*ffn*d/2) bytes:
 *             gate/up [2*ffn][d/2]  (rows [0,ffn) gate, [ffn,2*ffn) up),
 *             then down [d][ffn/2];
 *           low nibble of a byte = even element, high nibble = odd element.
 *   scales: expert j starts at j * (3*ffn*d/32) bytes:
 *             gate/up [2*ffn][d/32], then down [d][ffn/32].
 *   The shared expert (ffn = shared_ffn) follows expert n_experts-1 in both.
 *
 * Errors: every call returns 0 (MOE_OK) or a negative MOE_ERR_* code; the text
 * of the last error of a context is available from moe_last_error(). No call
 * aborts the process, traps the GPU or waits without a bound on the device.
 * A context is not thread-safe: calls on one context must not overlap, and two
 * forwards on one context must not run concurrently on different streams
 * (they share the context's workspace).
 */
#ifndef MOE_GB300_H
#define MOE_GB300_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

enum {
  MOE_OK = 0,
  MOE_ERR_INVALID_ARG = -1, /* a size, pointer or config field out of range */
  MOE_ERR_T_TOO_LARGE = -2, /* T > t_max of the context */
  MOE_ERR_NOT_LOADED = -3,  /* forward before both loads completed */
  MOE_ERR_CUDA = -4,        /* a CUDA runtime call failed (text in moe_last_error) */
  MOE_ERR_TIMEOUT = -5,     /* a bounded device-side wait gave up (status word) */
  MOE_ERR_NAN_SCALE = -6,   /* an E8M0 scale byte 0xFF (NaN) in the loaded experts */
  MOE_ERR_NOMEM = -7        /* a device or host allocation failed at create time */
};

enum { MOE_OUT_BF16 = 0, MOE_OUT_F32 = 1 };

/* moe_config.flags bits.
 * MOE_FLAG_TEST_FORCE_TIMEOUT exists for failure-detection tests only: one
 *   device-side wait of every single-launch forward (T <= 16) waits for a
 *   value no launch writes and gives up after 2 ms, so the forward completes
 *   with MOE_ERR_TIMEOUT in the status word (its output is then undefined).
 * MOE_FLAG_GENERAL_PATH makes every forward take the multi-kernel path (for
 *   testing both paths on the same shapes).
 * Weights and paths. A context stores its experts once (made at load time,
 *   lossless). If t_max * top_k > 16 and the shared-memory tables fit
 *   (n_experts up to 512) the layout is that of the block-scaled tcgen05 MMAs
 *   (MXFP4 weights x MXFP8 planes of x and of h): forwards with T <= 16 run as
 *   one launch (the fused tcgen05 kernel), larger T on the multi-kernel path
 *   with the tcgen05 GEMMs. Otherwise (every call a few tokens) it is the
 *   packed tile layout of the fused mma.sync kernel, which serves T <= 16 (and
 *   the register-decode tensor-core GEMMs larger T). MOE_FLAG_TC_GATEUP forces
 *   the tcgen05 layout (an error if the tables do not fit); MOE_FLAG_NO_TC
 *   forces the packed one. Within each path a token's
 *   output bits do not depend on the other tokens of its call; results agree
 *   within the bf16 and fp32 tolerances across paths. */
enum { MOE_FLAG_TEST_FORCE_TIMEOUT = 1u, MOE_FLAG_GENERAL_PATH = 2u, MOE_FLAG_TC_GATEUP = 4u, MOE_FLAG_NO_TC = 8u };

typedef struct moe_config {
  int d;          /* hidden size; a multiple of 32 */
  int ffn;        /* routed expert intermediate size; a multiple of 32 */
  int n_experts;  /* E, 1..512 */
  int top_k;      /* k, 1..min(E, 32) */
  int shared_ffn; /* shared expert intermediate size (multiple of 32), 0 = none */
  int t_max;      /* largest T a forward will be given; sizes the workspace */
  int out_dtype;  /* MOE_OUT_BF16 (bf16, round to nearest even) or MOE_OUT_F32 */
  unsigned flags; /* MOE_FLAG_* bits; 0 for normal use */
  /* Expert-parallel shard: this context holds and computes routed experts
   * [expert_begin, expert_end) only, and the shared expert only if
   * expert_begin == 0; both 0 (the default) means every expert. Routing still
   * runs over all n_experts (the router is replicated) and the routing
   * exports stay global; the output is this shard's part of y -- its pairs'
   * gate-weighted rows (and the shared expert on the first shard) -- so the
   * fp32 outputs (MOE_OUT_F32) of a set of shards that partition the experts
   * add up to the layer, in any fixed order. The pages run the layer on one
   * GPU or as one pipeline stage per GPU ("NInfer" Qwen3.8-Flash-Next notes,
   * the multi-GPU run line); sharding by experts is this library's plan for
   * several GPUs, with the exchange of x and of the partial outputs left to
   * the caller. */
  int expert_begin, expert_end;
  /* Expert weight format: MOE_FORMAT_MXFP4 (0, the default) or
   * MOE_FORMAT_AFFINE64 (affine group-64 experts, loaded by
   * moe_load_experts_affine), with weight_bits its code width (2, 3, 4 or 8;
   * ignored for MXFP4). Affine contexts need d, ffn and shared_ffn multiples
   * of 64, take the multi-kernel path for every T and reject
   * MOE_FLAG_TC_GATEUP. */
  int weight_format;
  int weight_bits;
} moe_config;

enum { MOE_FORMAT_MXFP4 = 0, MOE_FORMAT_AFFINE64 = 1 };

typedef struct moe_ctx moe_ctx;

/* Create a context for one MoE layer of the shape cfg gives ("Neural Server"
 * technical page, "What it runs on and what it runs": 128 experts, four
 * active per token, hidden 2880, per-expert MXFP4 weights; "Running
 * Qwen3.8-Flash-Next on a 32 GB Mac with Transformers", architecture: one
 * shared expert beside the routed ones) on CUDA device `device`. Allocates all
 * device memory the layer will ever use (weights in the library's packed
 * layout, router, and a workspace sized for t_max); no later call allocates.
 * Sets the per-device attributes of the library's kernels on `device`. On
 * success *out holds the context (owned by the caller, freed by moe_destroy);
 * on failure *out is NULL, nothing is left allocated, and the return code
 * says why: MOE_ERR_INVALID_ARG (a config field out of range),
 * MOE_ERR_NOMEM (a device allocation failed), MOE_ERR_CUDA. */
int moe_create(const moe_config* cfg, int device, moe_ctx** out);

/* Copy the router of the layer ("Neural Server" technical page, "How one
 * token and one prompt are processed": the router and top-k step that turn a
 * token's hidden state into expert ids and weights): w is fp32
 * [n_experts][d] row-major, bias is fp32 [n_experts] or NULL (no bias). Host
 * or device pointers (cudaMemcpyDefault); the caller keeps ownership of both.
 * Synchronous. Errors: MOE_ERR_INVALID_ARG (w NULL), MOE_ERR_CUDA. */
int moe_load_router(moe_ctx* ctx, const float* w, const float* bias);

/* Copy the shared expert's gate row -- the "shared_expert_gate" of the MoE
 * blocks in "Running Qwen3.8-Flash-Next on a 32 GB Mac with Transformers"
 * (its table of MoE blocks), held on the GPU as one fp32 row of the hidden
 * size per layer ("Nebula", table of GPU-resident components): w is fp32 [d],
 * a host or device pointer the caller keeps; NULL removes the gate. With a
 * gate row the shared expert's output of token t is scaled by
 * sigmoid(w . x_t), the dot product summed as a double-float (the pages name
 * the tensor, not the formula: the sigmoid of a one-row projection is the
 * plainest reading of a per-token gate); without one it is added with weight
 * 1. Synchronous. Errors: MOE_ERR_INVALID_ARG (the context has no shared
 * expert), MOE_ERR_CUDA. */
int moe_load_shared_gate(moe_ctx* ctx, const float* w);

/* Copy all experts the context holds (canonical layout above: its routed
 * experts expert_begin .. expert_end - 1 in order, then the shared expert if
 * it has it; host or device pointers, still owned by the caller) and repack them on the device into the library's tile
 * layout. The "Neural Server" technical page keeps its expert store the same
 * way ("A 117B-parameter model on one gaming PC": a byte-exact repack of the
 * checkpoint's MXFP4 tensors; "What it runs on and what it runs": 13,219,200 B
 * per expert). The repack is lossless: every code and scale byte is kept,
 * only their order changes. Synchronous; uses a temporary
 * staging buffer that it frees before returning. Errors: MOE_ERR_INVALID_ARG
 * (a NULL pointer), MOE_ERR_NAN_SCALE (a scale byte 0xFF, the OCP MX NaN;
 * the context then counts as not loaded), MOE_ERR_NOMEM, MOE_ERR_CUDA. */
int moe_load_experts(moe_ctx* ctx, const uint8_t* codes, const uint8_t* scales);

/* Copy all experts of an affine context (weight_format MOE_FORMAT_AFFINE64)
 * and repack them on the device -- the second expert format of the pages:
 * "Running Qwen3.8-Flash-Next on a 32 GB Mac with Transformers", the table of
 * where every weight lives (3-bit affine experts, group 64, 2.15 MB per
 * expert) and the notes under the decode table (a 16-bit scale and bias per
 * 64 weights). Weight = scale * q + bias, q an unsigned weight_bits-bit code.
 * `experts` holds the routed experts the context holds, in order, then the
 * shared expert if it has it; each expert (ffn f) in the canonical affine
 * layout of affine_expert_bytes(d, f, bits) = 3 f d bits / 8 + 3 f d / 16
 * bytes:
 *   codes of the gate/up rows [2f][d] (gate rows 0..f-1, up rows f..2f-1),
 *     then of the down rows [d][f]; each row one little-endian bit stream,
 *     element c at bits [bits c, bits c + bits) of it;
 *   bf16 scales of gate/up [2f][d/64], then of down [d][f/64];
 *   bf16 biases in the same order.
 * Host or device pointer, owned by the caller; the repack is lossless (every
 * code, scale and bias kept, only the order changes). Synchronous; uses a
 * temporary staging buffer that it frees before returning. Errors:
 * MOE_ERR_INVALID_ARG (NULL, or not an affine context), MOE_ERR_NAN_SCALE (a
 * scale or bias that is Inf or NaN; the context then counts as not loaded),
 * MOE_ERR_NOMEM, MOE_ERR_CUDA. moe_load_experts on an affine context returns
 * MOE_ERR_INVALID_ARG. */
int moe_load_experts_affine(moe_ctx* ctx, const uint8_t* experts);

/* Run the layer on T tokens (0 <= T <= t_max): every step of the formula at
 * the top of this file, in the pages' order --
 *   router logits and top-k with softmax gates: "Neural Server" technical
 *     page, "How one token and one prompt are processed" (4 ids and 4
 *     weights per token); "NInfer" Qwen3.8-Flash-Next notes, MoE execution
 *     (weights renormalised per token);
 *   grouping of the (token, expert) pairs by expert: "NInfer" notes, MoE
 *     execution; "Neural Server", "Prompt processing" (tokens grouped by
 *     expert on the GPU);
 *   gate/up, SiLU(gate) * up, down per pair: "NInfer" notes, MoE execution
 *     (fused gate/up kernel, then down); "Neural Server", "Prompt processing"
 *     (SwiGLU epilogue);
 *   the shared expert: "Running Qwen3.8-Flash-Next on a 32 GB Mac with
 *     Transformers", architecture;
 *   the gate-weighted combine in a fixed order: "NInfer" notes, MoE execution
 *     (outputs summed independently of the order experts finish in).
 * x: bf16 [T][d] row-major in device memory; out: [T][d] row-major in device
 * memory, bf16 or fp32 as the config says; both 16-byte aligned and owned by
 * the caller. stream: a cudaStream_t (NULL = the legacy default stream).
 * Asynchronous and stream-ordered: only enqueues kernels, performs no host
 * synchronisation and no allocation, so it may be captured in a CUDA graph.
 * Errors (returned at once, nothing enqueued): MOE_ERR_INVALID_ARG,
 * MOE_ERR_T_TOO_LARGE, MOE_ERR_NOT_LOADED, MOE_ERR_CUDA (launch failed).
 * Device-side failures are reported by moe_get_status after synchronising. */
int moe_forward(moe_ctx* ctx, const void* x, int T, void* out, void* stream);

/* moe_forward (same passages) with HOST buffers: enqueues the copy of x
 * (host, bf16 [T][d]) into the context, the layer, and the copy of the result
 * back to out (host) on `stream`. With synchronize != 0 it waits for the stream before returning;
 * with 0 the caller synchronises before reading out or reusing x. Pinned host
 * memory is needed for the copies to be asynchronous; pageable works too.
 * Page-locked buffers mapped into the device's address space (cudaHostAlloc /
 * cudaMallocHost, torch pin_memory) skip the staging copies: the kernels
 * write y straight into such an out_host, and a call that runs a
 * single-launch kernel (moe_launches_per_forward == 1) on at most 16 KB of x
 * also reads x straight from such an x_host (every CTA of those kernels
 * stages all of x, so larger x is faster through the copy; so is an x that
 * shares bytes with out). Same bytes, same result bits.
 * Each context has one staging buffer: do not overlap two calls on a context. */
int moe_forward_host(moe_ctx* ctx, const void* x_host, int T, void* out_host, void* stream, int synchronize);

/* Debug export of the last forward's routing and bucketing ("Neural Server"
 * technical page, "How one token and one prompt are processed": expert ids
 * and weights per token; "NInfer" notes, MoE execution: pairs grouped by
 * expert). Device or host pointers owned by the caller, any may be NULL:
 * ids int32 [T][k], gates fp32 [T][k], counts int32 [E], offsets int32 [E+1]
 * (exclusive prefix sum of counts), perm int32 [T*k] (pair p = t*k + j,
 * stably sorted by expert), inv int32 [T*k] (inv[perm[q]] = q: the row of
 * pair p in expert order). Stream-ordered after the forward on the same
 * stream; the caller synchronises before reading host copies. Errors:
 * MOE_ERR_INVALID_ARG (ctx NULL), MOE_ERR_CUDA (a copy failed). */
int moe_get_routing(moe_ctx* ctx, int32_t* ids, float* gates, int32_t* counts, int32_t* offsets, int32_t* perm,
                    int32_t* inv, void* stream);

/* Debug export of the last forward's router logits (the router of
 * moe_load_router) as an unevaluated sum of two fp32 numbers, logit = hi +
 * lo: hi, lo fp32 [T][E], device or host pointers owned by the caller. The single-kernel
 * path (T <= 16) and the multi-kernel path with T <= 32 compute every logit as
 * a double-float sum (hi = fl(logit)). The multi-kernel path with T > 32
 * computes every logit in fp32 with an error bound and the double-float sum
 * only for the experts that bound cannot rule out of the top k: those hold
 * hi + lo as above, the others their fp32 value and lo = 0. */
int moe_get_logits(moe_ctx* ctx, float* hi, float* lo, void* stream);

/* Device status word of the context (0 = fine, else a MOE_ERR_* code set by a
 * kernel, e.g. MOE_ERR_TIMEOUT when a bounded device-side wait gave up). No
 * page has a counterpart: it is the library's failure report. Synchronises
 * the context's device; clears the word when `clear` is nonzero. Returns the
 * word, or MOE_ERR_INVALID_ARG / MOE_ERR_CUDA if it cannot be read. */
int moe_get_status(moe_ctx* ctx, int clear);

/* Tracing hook. Registers n_events cudaEvent_t handles (created by the
 * caller) that every later moe_forward records on its stream at its phase
 * boundaries: event i just before phase i starts and event n_phases after the
 * last phase, where the phases are those moe_forward_phases() names. Pass
 * NULL / 0 to stop recording. n_events must be 0 or n_phases + 1. */
int moe_profile_events(moe_ctx* ctx, void* const* events, int n_events);

/* Number of phases of a forward of T tokens, and (if names != NULL) a
 * pointer to a static, comma-separated list of their names. */
int moe_forward_phases(const moe_ctx* ctx, int T, const char** names);

/* Number of kernels one moe_forward of T tokens launches. */
int moe_launches_per_forward(const moe_ctx* ctx, int T);

/* Routing without any allocation, for callers that cannot call cudaMalloc
 * (for example code running under an allocator that owns all device memory,
 * or inside a region where allocation is forbidden). No counterpart on the
 * pages: it is a packaging of the router, top-k and counting-sort steps above.
 *
 * Computes, for T tokens, the router logits (double-float), the top-k ids and
 * softmax gates, and the counting sort of the T*top_k pairs by expert -- the
 * same kernels and results as the routing of moe_forward's multi-kernel path.
 * The caller passes device pointers: x bf16 [T][d] and w_router fp32
 * [n_experts][d] (both 16-byte aligned), bias fp32 [n_experts] or NULL, and
 * the outputs ids int32 [T][top_k], gates fp32 [T][top_k], counts int32
 * [n_experts], offsets int32 [n_experts+1], perm int32 [T*top_k].
 * The scratch is one static 3 MiB device array that every device loading the
 * library holds until exit; sizes beyond it (T*n_experts > 65536 or
 * T*top_k > 32768) are rejected with MOE_ERR_INVALID_ARG. The array keeps the
 * last call's contents and is shared by all calls: calls whose kernels
 * overlap on the GPU (other streams, other threads) race. The first call on
 * each device looks the array up (with that device current); make that first
 * call before any stream capture. Uses the current device; asynchronous on
 * `stream`. Error text: moe_last_error(NULL) does not cover this call, use
 * moe_route_static_error(). */
int moe_route_static(const void* x, int T, int d, const float* w_router, const float* bias, int n_experts, int top_k,
                     int32_t* ids, float* gates, int32_t* counts, int32_t* offsets, int32_t* perm, void* stream);

/* Text of the calling thread's last error returned by moe_route_static (""
 * if none). The string belongs to the library and stays valid until that
 * thread's next failing moe_route_static call. */
const char* moe_route_static_error(void);

/* Measured rate of the block-scaled tensor-core MMA the expert GEMMs issue
 * (tcgen05.mma kind::mxf8f6f4: E2M1 weights x E4M3 activations with UE8M0
 * scales, M = 128, K = 32, N = n: a multiple of 16 in [16, 192]) on CUDA
 * device `device`. No page has a
 * counterpart: it measures this GPU, as the denominator of the GEMMs'
 * tensor-pipe fraction. One CTA per SM issues mmas_per_sm MMAs back to back
 * from shared-memory operands (no memory traffic) into tensor memory; the
 * call times one such launch with CUDA events after a warm-up launch and
 * returns the dense rate in *tflops (10^12 multiply-adds x 2 per second) and
 * the launch time in *ms (may be NULL). Synchronous; allocates and frees a
 * 4-byte status word and two events. Errors: MOE_ERR_INVALID_ARG
 * (mmas_per_sm outside [1, 2^24], n not as above, or tflops NULL), MOE_ERR_CUDA,
 * MOE_ERR_TIMEOUT (the MMAs did not finish within 2 s); text from
 * moe_probe_error(). */
int moe_probe_mma_rate(int device, int mmas_per_sm, int n, double* tflops, double* ms);

/* Text of the calling thread's last error returned by moe_probe_mma_rate. */
const char* moe_probe_error(void);

/* Bytes of expert weights the context holds in its layout (codes + scales:
 * the packed tiles, exactly the canonical size, or the tcgen05 blocks, the
 * canonical size plus the zero padding of partial 128-row tiles; the "Neural
 * Server" technical page, "What it runs on and what it runs", counts
 * 13,219,200 B per gpt-oss-120B expert). 0 for a NULL ctx. */
size_t moe_weight_bytes(const moe_ctx* ctx);

/* Text of the last error raised on this context ("" if none); no page has a
 * counterpart. NULL ctx gives the text of the last failed moe_create. The
 * string belongs to the context and stays valid until its next failing call
 * or moe_destroy. */
const char* moe_last_error(const moe_ctx* ctx);

/* Free everything the context owns (weights, router, workspace). NULL is
 * accepted. The caller must not have work of this context in flight. */
void moe_destroy(moe_ctx* ctx);

#ifdef __cplusplus
}
#endif

#endif /* MOE_GB300_H */
