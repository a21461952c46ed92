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
 *   device-side wait of every single-kernel decode forward waits for a value
 *   no launch writes and gives up after 2 ms, so the forward completes with
 *   MOE_ERR_TIMEOUT in the status word (its output is then undefined).
 * MOE_FLAG_GENERAL_PATH makes every forward take the multi-kernel path (for
 *   testing both paths on the same shapes).
 * Path choice per call: the fused single-kernel path serves T <= 16 unless
 *   the context holds the tcgen05 weight copy and T * top_k > 16; every other
 *   call takes the multi-kernel path. Within each class a token's output bits
 *   do not depend on the other tokens of its call.
 * The multi-kernel path runs both expert GEMMs as block-scaled tcgen05 MMAs
 *   (MXFP4 weights x MXFP8 planes of x and of h) from a second copy of the
 *   experts in the MMA's layout, made at load time, whenever t_max * top_k >
 *   16 and the shared-memory tables fit (n_experts up to 512).
 * MOE_FLAG_TC_GATEUP asks for those MMAs for every t_max (an error if the
 *   tables do not fit); MOE_FLAG_NO_TC keeps the register-decode tensor-core
 *   GEMMs instead (no second copy; T <= 16 then always takes the fused
 *   path). Results agree within the bf16 and fp32 tolerances either way. */
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
} moe_config;

typedef struct moe_ctx moe_ctx;

/* Create a context on CUDA device `device`. Allocates all device memory the
 * layer will ever use (weights in the library's packed layout, router, and a
 * workspace sized for t_max); no later call allocates. On success *out holds
 * the context; on failure *out is NULL and the return code says why. */
int moe_create(const moe_config* cfg, int device, moe_ctx** out);

/* Copy the router: w is fp32 [n_experts][d] row-major, bias is fp32
 * [n_experts] or NULL (no bias). Host or device pointers (cudaMemcpyDefault).
 * Synchronous. Section: "Neural Server", "How one token ... processed". */
int moe_load_router(moe_ctx* ctx, const float* w, const float* bias);

/* Copy all experts (canonical layout above; host or device pointers) and
 * repack them on the device into the library's tile layout. The repack is
 * lossless: every code and scale byte is kept, only their order changes.
 * Synchronous. Returns MOE_ERR_NAN_SCALE if any scale byte is 0xFF. */
int moe_load_experts(moe_ctx* ctx, const uint8_t* codes, const uint8_t* scales);

/* Run the layer on T tokens (0 <= T <= t_max). x: bf16 [T][d] row-major in
 * device memory; out: [T][d] row-major in device memory, bf16 or fp32 as the
 * config says. stream: a cudaStream_t (NULL = the legacy default stream).
 * Asynchronous and stream-ordered: only enqueues kernels, performs no host
 * synchronisation and no allocation, so it may be captured in a CUDA graph.
 * Device-side failures are reported by moe_get_status after synchronising. */
int moe_forward(moe_ctx* ctx, const void* x, int T, void* out, void* stream);

/* moe_forward with HOST buffers: enqueues the copy of x (host, bf16 [T][d])
 * into the context, the layer, and the copy of the result back to out (host)
 * on `stream`. With synchronize != 0 it waits for the stream before returning;
 * with 0 the caller synchronises before reading out or reusing x. Pinned host
 * memory is needed for the copies to be asynchronous; pageable works too.
 * Each context has one staging buffer: do not overlap two calls on a context. */
int moe_forward_host(moe_ctx* ctx, const void* x_host, int T, void* out_host, void* stream, int synchronize);

/* Debug export of the last forward's routing (device or host pointers, any
 * may be NULL): ids int32 [T][k], gates fp32 [T][k], counts int32 [E],
 * offsets int32 [E+1], perm int32 [T*k] (pair p = t*k + j, stably sorted by
 * expert). Stream-ordered after the forward on the same stream; the caller
 * synchronises before reading host copies. */
int moe_get_routing(moe_ctx* ctx, int32_t* ids, float* gates, int32_t* counts, int32_t* offsets, int32_t* perm,
                    void* stream);

/* Debug export of the last forward's router logits as an unevaluated sum of
 * two fp32 numbers, logit = hi + lo: hi, lo fp32 [T][E]. The single-kernel
 * path (T <= 16) and the multi-kernel path with T <= 32 compute every logit as
 * a double-float sum (hi = fl(logit)). The multi-kernel path with T > 32
 * computes every logit in fp32 with an error bound and the double-float sum
 * only for the experts that bound cannot rule out of the top k: those hold
 * hi + lo as above, the others their fp32 value and lo = 0. */
int moe_get_logits(moe_ctx* ctx, float* hi, float* lo, void* stream);

/* Device status word of the context (0 = fine, else a MOE_ERR_* code set by a
 * kernel, e.g. MOE_ERR_TIMEOUT). Synchronises the context's device; clears the
 * word when `clear` is nonzero. */
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

/* Text of the last error returned by moe_route_static ("" if none). */
const char* moe_route_static_error(void);

/* Bytes of packed expert weights the context holds (codes + scales). */
size_t moe_weight_bytes(const moe_ctx* ctx);

/* Text of the last error raised on this context ("" if none). NULL ctx gives
 * the text of the last failed moe_create. */
const char* moe_last_error(const moe_ctx* ctx);

/* Free everything the context owns. NULL is accepted. */
void moe_destroy(moe_ctx* ctx);

#ifdef __cplusplus
}
#endif

#endif /* MOE_GB300_H */
