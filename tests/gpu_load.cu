// Test helper: a background load that holds SMs while a GEMM runs on another
// stream.  Each CTA takes 96 KiB of shared memory (so no GEMM CTA fits beside
// it) and spins on the global timer for a fixed time: it always ends.
#include <cuda_runtime.h>
#include <stdint.h>

__global__ void hold_sms_kernel(uint64_t ns) {
  extern __shared__ char pad[];
  uint64_t t0, t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t0));
  do {
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  } while (t - t0 < ns);
  if (threadIdx.x == 0 && t == 0) pad[0] = 1;  // keeps the allocation
}

extern "C" int hold_sms(int ctas, unsigned long long ns, void* stream) {
  cudaError_t e = cudaFuncSetAttribute(hold_sms_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, 96 * 1024);
  if (e != cudaSuccess) return (int)e;
  hold_sms_kernel<<<ctas, 32, 96 * 1024, (cudaStream_t)stream>>>(ns);
  return (int)cudaGetLastError();
}
