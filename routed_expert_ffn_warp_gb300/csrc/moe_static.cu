// Routing entry point that allocates nothing: its scratch (router logits,
// sums of squares and the bucketing work list) lives in one file-scope device
// array of fixed size instead of memory obtained from cudaMalloc.
#include <cuda_runtime.h>

#include <cstdint>
#include <mutex>
#include <string>

#include "../../include/moe.h"
#include "moe_internal.h"

namespace {

constexpr size_t kScratchBytes = size_t(3) << 20;  // 3 MiB on every device that loads the library
constexpr size_t kMaxLogits = 65536;              // T * n_experts
constexpr size_t kMaxPairs = 32768;               // T * top_k
constexpr int kMaxDevices = 64;

// Layout of the scratch array (byte offsets): the router's partial-logit
// planes (the first two are the logits' hi and lo), inverse permutation,
// work-list slots, sums of squares of the router rows and of x (these are
// fully rewritten by every call; no part must start at zero).
constexpr int kStaticSplits = 4;  // ranges of d of the router's fp32 pass this array has planes for
constexpr size_t kOffHi = 0;
constexpr size_t kOffInv = kOffHi + kStaticSplits * kMaxLogits * 4;
constexpr size_t kOffSlots = kOffInv + kMaxPairs * 4;
constexpr size_t kSlotInts = 1 + 3 * 513 + 2 * 514;
constexpr size_t kOffWsq = (kOffSlots + kSlotInts * 4 + 255) / 256 * 256;
constexpr size_t kOffXsq = kOffWsq + kStaticSplits * 512 * 4;
static_assert(kOffXsq + kStaticSplits * kMaxLogits * 4 <= kScratchBytes, "scratch layout exceeds the array");

__device__ __align__(256) unsigned char g_route_scratch[kScratchBytes];

std::mutex g_mu;                   // guards g_scratch
void* g_scratch[kMaxDevices] = {};  // device address of g_route_scratch, per device
// Error text of the calling thread's last failed call: one string per thread,
// so the pointer moe_route_static_error hands out is never rewritten by
// another thread's failure.
thread_local std::string t_err;

int fail(int code, const std::string& msg) {
  t_err = msg;
  return code;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

}  // namespace

extern "C" const char* moe_route_static_error(void) { return t_err.c_str(); }

extern "C" int moe_route_static(const void* x, int T, int d, const float* w_router, const float* bias, int n_experts,
                                int top_k, int32_t* ids, float* gates, int32_t* counts, int32_t* offsets,
                                int32_t* perm, void* stream) {
  if (T < 0 || d <= 0 || d % 32 || n_experts < 1 || n_experts > 512 || top_k < 1 || top_k > n_experts || top_k > 32)
    return fail(MOE_ERR_INVALID_ARG, "moe_route_static: need T >= 0, d a multiple of 32, 1 <= n_experts <= 512, "
                                     "1 <= top_k <= min(n_experts, 32)");
  if ((size_t)T * (size_t)n_experts > kMaxLogits || (size_t)T * (size_t)top_k > kMaxPairs)
    return fail(MOE_ERR_INVALID_ARG, "moe_route_static: T * n_experts must be <= 65536 and T * top_k <= 32768 "
                                     "(the static scratch holds 3 MiB)");
  if (T == 0) return MOE_OK;
  if (!x || !w_router || !ids || !gates || !counts || !offsets || !perm)
    return fail(MOE_ERR_INVALID_ARG, "moe_route_static: a required pointer is NULL");
  if (!aligned16(x) || !aligned16(w_router))
    return fail(MOE_ERR_INVALID_ARG, "moe_route_static: x and w_router must be 16-byte aligned");
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return fail(MOE_ERR_CUDA, std::string("cudaGetDevice: ") + cudaGetErrorString(e));
  if (dev < 0 || dev >= kMaxDevices) return fail(MOE_ERR_INVALID_ARG, "moe_route_static: device index too large");
  void* base = nullptr;
  {
    std::lock_guard<std::mutex> lk(g_mu);
    if (!g_scratch[dev]) {
      // first call on this device (its device is current): look the array up once
      e = cudaGetSymbolAddress(&g_scratch[dev], g_route_scratch);
      if (e != cudaSuccess) {
        g_scratch[dev] = nullptr;
        return fail(MOE_ERR_CUDA, std::string("cudaGetSymbolAddress: ") + cudaGetErrorString(e));
      }
    }
    base = g_scratch[dev];
  }
  char* sc = static_cast<char*>(base);
  moe::FwdParams p{};
  p.T = T;
  p.d = d;
  p.E = n_experts;
  p.e_begin = 0;
  p.e_end = n_experts;
  p.k = top_k;
  p.F = 0;
  p.S = 0;
  p.P = T * top_k;
  p.x = static_cast<const uint16_t*>(x);
  p.w_router = w_router;
  p.bias = bias;
  p.logit_hi = reinterpret_cast<float*>(sc + kOffHi);
  p.lstride = (size_t)T * n_experts;
  p.rsplit_max = kStaticSplits;
  p.logit_lo = p.logit_hi + p.lstride;
  p.wsq = reinterpret_cast<float*>(sc + kOffWsq);
  p.xsq = reinterpret_cast<float*>(sc + kOffXsq);
  p.ids = ids;
  p.gates = gates;
  p.counts = counts;
  p.offsets = offsets;
  p.perm = perm;
  p.inv = reinterpret_cast<int32_t*>(sc + kOffInv);
  int32_t* slots = reinterpret_cast<int32_t*>(sc + kOffSlots);
  p.n_slots = slots;
  p.slot_expert = slots + 1;
  p.slot_q0 = p.slot_expert + 513;
  p.slot_n = p.slot_q0 + 513;
  p.gu_prefix = p.slot_n + 513;
  p.dn_prefix = p.gu_prefix + 514;
  // the bucketing kernel's shared-memory limit is a per-device attribute (no context sets it here)
  if ((e = moe::configure_kernels()) != cudaSuccess)
    return fail(MOE_ERR_CUDA, std::string("moe_route_static: ") + cudaGetErrorString(e));
  e = moe::launch_route(p, static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return fail(MOE_ERR_CUDA, std::string("moe_route_static launch: ") + cudaGetErrorString(e));
  return MOE_OK;
}
