// Measured rate of the block-scaled tensor-core MMA that the expert GEMMs of
// this library issue: tcgen05.mma kind::mxf8f6f4 with E2M1 weights, E4M3
// activations and UE8M0 scale factors, M = 128, K = 32 and N = 16 .. 192 (a
// multiple of 16: the widths the gate/up and down GEMMs issue; 192 is the
// down GEMM's widest unit). Every SM runs one CTA whose single issuing
// thread sends MMAs back to back into one TMEM accumulator from operands that
// stay in shared memory, so the time is the tensor pipe's alone (no memory
// traffic). The rate is the denominator the prefill GEMMs' tensor-pipe
// fraction is reported against; no page has a counterpart (the pages name
// tensor-core kernels, not this GPU's rates).
#include <cuda_runtime.h>

#include <string>

#include "../../include/moe.h"
#include "moe_device.cuh"
#include "moe_internal.h"
#include "moe_tc.cuh"

namespace moe {
namespace {

using namespace dev;

constexpr int kProbeM = 128, kProbeMaxN = 192, kProbeK = 32;
constexpr int kProbeThreads = 128;          // four warps: one per TMEM lane quadrant for the scale stores
constexpr int kProbeA = 16 * 1024;          // A: 16 eight-row groups of 8 core matrices (1,024 bytes each)
constexpr int kProbeB = kProbeMaxN / 8 * 1024;  // B: up to 24 eight-row groups
constexpr uint32_t kProbeCols = 512;        // accumulator at column 0 (192 wide), scale factors at 384
constexpr int kProbeSf = 384;
constexpr long long kProbeWaitNs = 2000000000LL;  // 2 s: far above any probe length the host asks for

__global__ void __launch_bounds__(kProbeThreads, 1) mma_rate_kernel(int n_mma, int n, int* status) {
  extern __shared__ __align__(1024) uint8_t sm[];
  uint8_t* a = sm;
  uint8_t* b = sm + kProbeA;
  uint64_t* bar = reinterpret_cast<uint64_t*>(sm + kProbeA + kProbeB);
  uint32_t* tslot = reinterpret_cast<uint32_t*>(bar + 1);
  const int tid = threadIdx.x, warp = tid >> 5;
  // A: E2M1 code pairs 0x22 (1.0, 1.0) in the 8 code bytes of every 16-byte row, zero padding;
  // B: E4M3 0x38 (1.0). Finite values: the accumulator grows by 32 per MMA, far from overflow.
  for (int i = tid; i < kProbeA / 16; i += kProbeThreads)
    reinterpret_cast<uint4*>(a)[i] = make_uint4(0x22222222u, 0x22222222u, 0u, 0u);
  for (int i = tid; i < kProbeB / 4; i += kProbeThreads) reinterpret_cast<uint32_t*>(b)[i] = 0x38383838u;
  tc::fence_proxy_async();
  if (tid == 0) {
    mbar_init(bar, 1);
    fence_mbar_init();
  }
  if (warp == 0) tc::alloc(tslot, kProbeCols);
  tc::fence_before();
  __syncthreads();
  tc::fence_after();
  const uint32_t tmem = *tslot;
  // scale factors 2^0 (byte 127) in every lane quadrant: A rows 32 r + l in columns +0..+3, B rows in +16..+23
  const uint32_t q = tmem + ((uint32_t)((warp & 3) * 32) << 16) + kProbeSf;
  const uint32_t one = 0x7F7F7F7Fu;
  tc::st4(q, one, one, one, one);
  tc::st4(q + 16, one, one, one, one);
  tc::st4(q + 20, one, one, one, one);
  tc::wait_st();
  tc::fence_before();
  __syncthreads();
  tc::fence_after();
  if (tid == 0) {
    for (int i = 0; i < n_mma; ++i) {
      const int kb = i & 3;  // the four K = 32 blocks of the operand, each with its own scale-factor id
      const uint64_t ad = tc::smem_desc(a + 2 * kb * 128, 128, 8 * 128);
      const uint64_t bd = tc::smem_desc(b + 2 * kb * 128, 128, 8 * 128);
      tc::mma_mxf4_mxf8(tmem, ad, bd, tc::idesc_mxf4_mxf8(kProbeM, n, kb, kb), tmem + kProbeSf,
                        tmem + kProbeSf + 16, i > 0 ? 1u : 0u);
    }
    tc::commit(bar);
    const uint64_t t0 = globaltimer();
    while (!mbar_try_wait(bar, 0)) {
      if ((long long)(globaltimer() - t0) > kProbeWaitNs) {
        atomicCAS(status, 0, MOE_ERR_TIMEOUT);
        // the MMAs still hold tensor memory: give them time before it is freed
        const uint64_t t1 = globaltimer();
        while ((long long)(globaltimer() - t1) < 100000000LL) __nanosleep(100000);
        break;
      }
    }
  }
  tc::fence_before();
  __syncthreads();
  if (warp == 0) {
    tc::fence_after();
    tc::dealloc(tmem, kProbeCols);
  }
}

thread_local std::string t_probe_err;

int probe_fail(int code, const std::string& msg) {
  t_probe_err = msg;
  return code;
}

}  // namespace
}  // namespace moe

extern "C" const char* moe_probe_error(void) { return moe::t_probe_err.c_str(); }

extern "C" int moe_probe_mma_rate(int device, int mmas_per_sm, int n, double* tflops, double* ms) {
  using namespace moe;
  if (mmas_per_sm < 1 || mmas_per_sm > (1 << 24) || !tflops || n < 16 || n > kProbeMaxN || n % 16)
    return probe_fail(MOE_ERR_INVALID_ARG, "moe_probe_mma_rate: need 1 <= mmas_per_sm <= 2^24, n a multiple of 16 "
                                           "in [16, 192] and tflops != NULL");
  int prev = -1;
  if (cudaGetDevice(&prev) != cudaSuccess) prev = -1;
  if (prev != device && cudaSetDevice(device) != cudaSuccess)
    return probe_fail(MOE_ERR_CUDA, "moe_probe_mma_rate: cudaSetDevice failed");
  int rc = MOE_OK;
  int* status = nullptr;
  cudaEvent_t e0 = nullptr, e1 = nullptr;
  int sms = 0, max_smem = 0;
  float t_ms = 0.f;
  cudaError_t e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, device);
  if (e == cudaSuccess) e = cudaDeviceGetAttribute(&max_smem, cudaDevAttrMaxSharedMemoryPerBlockOptin, device);
  // more than half of an SM's shared memory: one CTA per SM, each with the whole TMEM
  const int smem = max_smem / 2 + 1024;
  if (e == cudaSuccess && smem < kProbeA + kProbeB + 64) e = cudaErrorInvalidValue;
  if (e == cudaSuccess) e = cudaFuncSetAttribute(mma_rate_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e == cudaSuccess) e = cudaMalloc(&status, sizeof(int));
  if (e == cudaSuccess) e = cudaMemset(status, 0, sizeof(int));
  if (e == cudaSuccess) e = cudaEventCreate(&e0);
  if (e == cudaSuccess) e = cudaEventCreate(&e1);
  if (e == cudaSuccess) {
    mma_rate_kernel<<<sms, kProbeThreads, smem>>>(1024, n, status);  // warm-up: clocks up, code loaded
    e = cudaGetLastError();
  }
  if (e == cudaSuccess) e = cudaEventRecord(e0);
  if (e == cudaSuccess) {
    mma_rate_kernel<<<sms, kProbeThreads, smem>>>(mmas_per_sm, n, status);
    e = cudaGetLastError();
  }
  if (e == cudaSuccess) e = cudaEventRecord(e1);
  if (e == cudaSuccess) e = cudaEventSynchronize(e1);
  if (e == cudaSuccess) e = cudaEventElapsedTime(&t_ms, e0, e1);
  int st = 0;
  if (e == cudaSuccess) e = cudaMemcpy(&st, status, sizeof(int), cudaMemcpyDeviceToHost);
  if (e != cudaSuccess) {
    rc = probe_fail(MOE_ERR_CUDA, std::string("moe_probe_mma_rate: ") + cudaGetErrorString(e));
  } else if (st != 0) {
    rc = probe_fail(st, "moe_probe_mma_rate: the MMAs did not complete within the bound");
  } else {
    const double flops = 2.0 * kProbeM * n * kProbeK * (double)mmas_per_sm * (double)sms;
    *tflops = flops / ((double)t_ms * 1e-3) / 1e12;
    if (ms) *ms = t_ms;
  }
  if (e0) cudaEventDestroy(e0);
  if (e1) cudaEventDestroy(e1);
  cudaFree(status);
  if (prev >= 0 && prev != device) cudaSetDevice(prev);
  return rc;
}
