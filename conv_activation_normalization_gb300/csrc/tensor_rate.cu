// Tensor-pipe rate probe: gf_measure_tensor_rate.
//
// One CTA per SM issues tcgen05.mma instructions back to back on operand
// tiles that already sit in shared memory (no loads, no epilogue): a 128 x 256
// fp32 accumulator in TMEM, four 32-byte K-steps of one 128-byte k-block per
// round, `iters` rounds.  Its rate is the tensor pipe's own rate for that
// operand kind on this GPU; the ratio of the TF32 and BF16 rates turns the
// measured cuBLAS BF16 peak into a measured TF32 (and 3xTF32-effective) peak.
#include <cstdint>

#include "host_common.h"
#include "ptx.cuh"

namespace gf {
namespace {

constexpr int kRateM = 128, kRateN = 256;
constexpr int kRateABytes = kRateM * 128, kRateBBytes = kRateN * 128;
constexpr int kRateSmem = kRateABytes + kRateBBytes + 1024 /*alignment*/ + 64 /*barrier, slot*/;

template <bool TF32>
__global__ void __launch_bounds__(128, 1) tensor_rate_kernel(int iters, uint32_t* status) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t* done = reinterpret_cast<uint64_t*>(smem + kRateABytes + kRateBBytes);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(done + 1);
  // operand values of moderate size (what they are does not matter, only
  // that they are ordinary finite numbers)
  for (int i = threadIdx.x; i < (kRateABytes + kRateBBytes) / 4; i += blockDim.x) {
    const float v = float(int((i * 2654435761u) >> 20) - 2048) * (1.f / 2048.f);
    if constexpr (TF32) {
      reinterpret_cast<float*>(smem)[i] = v;
    } else {
      const uint32_t h = __float_as_uint(v) >> 16;  // bf16 of v (truncated), twice
      reinterpret_cast<uint32_t*>(smem)[i] = h | (h << 16);
    }
  }
  fence_proxy_async_smem();
  if (threadIdx.x == 0) {
    mbar_init(done, 1);
    fence_mbar_init();
  }
  if (threadIdx.x < 32) {
    tmem_alloc(smem_u32(tmem_slot), kRateN);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  if (threadIdx.x == 0) {
    constexpr uint32_t idesc = TF32 ? idesc_tf32(kRateM, kRateN) : idesc_bf16(kRateM, kRateN);
    const uint32_t a = smem_u32(smem), b = a + kRateABytes;
    for (int it = 0; it < iters; ++it) {
#pragma unroll
      for (int kk = 0; kk < 4; ++kk) {
        const uint64_t ad = sdesc_kmajor_sw128(a + kk * 32), bd = sdesc_kmajor_sw128(b + kk * 32);
        if constexpr (TF32)
          mma_tf32(tmem, ad, bd, idesc, (it | kk) != 0);
        else
          mma_bf16(tmem, ad, bd, idesc, (it | kk) != 0);
      }
    }
    mma_commit(done);
    if (!mbar_wait(done, 0)) record_error(status, GF_DEV_WAIT_TIMEOUT);
  }
  tc_fence_before();
  __syncthreads();
  if (threadIdx.x < 32) {
    tc_fence_after();
    tmem_dealloc(tmem, kRateN);
  }
}

}  // namespace
}  // namespace gf

using namespace gf;

extern "C" {

gf_status gf_measure_tensor_rate(int32_t kind, int32_t iters, int32_t repeats, double* tflops) {
  if (!tflops) return GF_ERR_NULL;
  if ((kind != 0 && kind != 1) || iters < 1 || iters > (1 << 16) || repeats < 1 || repeats > 100)
    return GF_ERR_SHAPE;
  DeviceInfo dev;
  gf_status st = current_device(&dev);
  if (st != GF_OK) return st;
  auto kern = kind == 0 ? tensor_rate_kernel<true> : tensor_rate_kernel<false>;
  if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, kRateSmem) != cudaSuccess)
    return GF_ERR_CUDA;
  cudaStream_t s = nullptr;
  cudaEvent_t e0 = nullptr, e1 = nullptr;
  if (cudaStreamCreateWithFlags(&s, cudaStreamNonBlocking) != cudaSuccess) return GF_ERR_CUDA;
  if (cudaEventCreate(&e0) != cudaSuccess || cudaEventCreate(&e1) != cudaSuccess) {
    if (e0) cudaEventDestroy(e0);
    cudaStreamDestroy(s);
    return GF_ERR_CUDA;
  }
  // FLOP of one MMA instruction: 2 M N K, K = 32 bytes of fp32 (8) or bf16 (16)
  const double flop = double(dev.sm_count) * iters * 4 * 2.0 * kRateM * kRateN * (kind == 0 ? 8 : 16);
  double best = 0.0;
  for (int r = 0; r <= repeats && st == GF_OK; ++r) {  // launch 0 warms up
    cudaEventRecord(e0, s);
    kern<<<dev.sm_count, 128, kRateSmem, s>>>(iters, device_status_word());
    cudaEventRecord(e1, s);
    float ms = 0.f;
    if (cudaGetLastError() != cudaSuccess || cudaEventSynchronize(e1) != cudaSuccess ||
        cudaEventElapsedTime(&ms, e0, e1) != cudaSuccess)
      st = GF_ERR_CUDA;
    else if (r > 0 && ms > 0.f && flop / (ms * 1e-3) * 1e-12 > best)
      best = flop / (ms * 1e-3) * 1e-12;
  }
  cudaEventDestroy(e0);
  cudaEventDestroy(e1);
  cudaStreamDestroy(s);
  *tflops = best;
  return st;
}

}  // extern "C"
