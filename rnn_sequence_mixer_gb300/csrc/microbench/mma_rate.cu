// mma_rate.cu — tensor-core throughput of the prefill's MMA sequence with its
// operands resident in shared memory (libhla_mmabench.so, measurement only;
// not part of the C ABI of libhla.so).
//
// Each CTA (one per SM) holds the operand tiles of one 128-token tile and
// issues, iters times, the four MMAs of the output pass of tc_prefill.cu with
// their shapes, types and layouts: P = Q~ K~^T (fp16), O = Q~ Sb (fp16),
// O += Pm V (bf16), S += K~dec^T V (bf16), each 128 x 128 x 128.  Nothing else
// runs, so the rate is the ceiling of the tensor-core part of the pass.
#include <cuda.h>
#include <cuda_fp16.h>

#include "../hla_internal.cuh"
#include "../umma.cuh"

namespace {

constexpr int ROWS = 128, TILE = 128 * 128 * 2;

__device__ unsigned int g_status;

__global__ void __launch_bounds__(128, 1) mma_rate_kernel(int iters) {
  extern __shared__ unsigned char smem_raw[];
  unsigned char *base = (unsigned char *)(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
  // Q16, K16, S16 (fp16), Pm, V, Kd (bf16); then the barrier and the TMEM address
  uint64_t *bar = reinterpret_cast<uint64_t *>(base + 6 * TILE);
  uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(base + 6 * TILE + 8);
  const int tid = threadIdx.x;
  // small values (1/64) in every element, as fp16 bits in the first three tiles, bf16 after
  for (int e = tid; e < 6 * TILE / 4; e += blockDim.x) {
    const bool half = e < 3 * TILE / 4;
    reinterpret_cast<uint32_t *>(base)[e] = half ? 0x24002400u : 0x3c803c80u;
  }
  if (tid == 0) {
    hla::umma::mbar_init(bar, 1);
    hla::umma::mbar_fence_init();
  }
  if (tid < 32) hla::umma::tmem_alloc(tmem_slot, 512);
  hla::umma::fence_async_smem();
  hla::umma::fence_before();
  __syncthreads();
  hla::umma::fence_after();
  const uint32_t tm = *tmem_slot;
  if (tid == 0) {
    const uint32_t aq = hla::umma::smem_u32(base), ak = aq + TILE, as = aq + 2 * TILE;
    const uint32_t apm = aq + 3 * TILE, av = aq + 4 * TILE, akd = aq + 5 * TILE;
    constexpr uint32_t id_qk = hla::umma::idesc_bf16(128, 128, false, false, true);
    constexpr uint32_t id_qs = hla::umma::idesc_bf16(128, 128, false, true, true);
    constexpr uint32_t id_pv = hla::umma::idesc_bf16(128, 128, false, true);
    constexpr uint32_t id_mn = hla::umma::idesc_bf16(128, 128, true, true);
    for (int it = 0; it < iters; ++it) {
#pragma unroll
      for (int kk = 0; kk < 8; ++kk)
        hla::umma::mma_ss(tm, hla::umma::desc_kmajor(aq, kk, ROWS), hla::umma::desc_kmajor(ak, kk, ROWS),
                          id_qk, kk > 0);
#pragma unroll
      for (int kk = 0; kk < 8; ++kk)
        hla::umma::mma_ss(tm + 128, hla::umma::desc_kmajor(aq, kk, ROWS),
                          hla::umma::desc_mnmajor(as, kk, ROWS), id_qs, kk > 0);
#pragma unroll
      for (int kk = 0; kk < 8; ++kk)
        hla::umma::mma_ss(tm + 128, hla::umma::desc_kmajor(apm, kk, ROWS),
                          hla::umma::desc_mnmajor(av, kk, ROWS), id_pv, 1u);
#pragma unroll
      for (int kk = 0; kk < 8; ++kk)
        hla::umma::mma_ss(tm + 384, hla::umma::desc_mnmajor(akd, kk, ROWS),
                          hla::umma::desc_mnmajor(av, kk, ROWS), id_mn, it > 0 || kk > 0);
    }
    hla::umma::commit(bar);
    if (!hla::umma::mbar_wait(bar, 0)) atomicOr(&g_status, 1u);
  }
  hla::umma::fence_before();
  __syncthreads();
  hla::umma::fence_after();
  if (tid < 32) hla::umma::tmem_dealloc(tm, 512);
}

}  // namespace

// Runs the kernel on `ctas` CTAs for `iters` iterations each and reports the
// elapsed device time in *ms (CUDA events around the launch, after one
// warm-up launch).  Returns 0 on success, 1 if a bounded wait gave up, -1 on a
// CUDA error.
extern "C" int hla_mmabench_run(int ctas, int iters, float *ms) {
  const size_t smem = 6 * TILE + 64 + 1024;
  if (ctas < 1 || iters < 1 || !ms) return -1;
  if (cudaFuncSetAttribute(mma_rate_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           (int)smem) != cudaSuccess)
    return -1;
  unsigned int zero = 0;
  if (cudaMemcpyToSymbol(g_status, &zero, sizeof(zero)) != cudaSuccess) return -1;
  cudaEvent_t a, b;
  cudaEventCreate(&a);
  cudaEventCreate(&b);
  mma_rate_kernel<<<ctas, 128, smem>>>(iters);  // warm-up
  cudaEventRecord(a);
  mma_rate_kernel<<<ctas, 128, smem>>>(iters);
  cudaEventRecord(b);
  const cudaError_t e = cudaEventSynchronize(b);
  cudaEventElapsedTime(ms, a, b);
  cudaEventDestroy(a);
  cudaEventDestroy(b);
  if (e != cudaSuccess || cudaGetLastError() != cudaSuccess) return -1;
  unsigned int status = 0;
  cudaMemcpyFromSymbol(&status, g_status, sizeof(status));
  return status ? 1 : 0;
}
