// Test helper (not part of the library): a kernel whose blocks each hold one SM
// for a bounded time, so a test can run the library's kernels on the SMs that
// are left. Each block takes `smem` bytes of shared memory (enough that no
// 200 KB CTA fits beside it) and spins on the global timer until `ns` have
// passed; `started` counts the blocks that are running.
#include <cuda_runtime.h>

__global__ void occupy_kernel(unsigned long long ns, int* started) {
  extern __shared__ unsigned char buf[];
  unsigned long long t0, t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t0));
  if (threadIdx.x == 0) atomicAdd(started, 1);
  buf[threadIdx.x] = (unsigned char)threadIdx.x;
  do {
    __nanosleep(1000);
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  } while (t - t0 < ns);
  if (buf[threadIdx.x] != (unsigned char)threadIdx.x) atomicAdd(started, 1000000);
}

extern "C" int occupy_sms(int blocks, unsigned long long ns, int smem, int* started, cudaStream_t st) {
  cudaError_t e = cudaFuncSetAttribute(occupy_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return (int)e;
  occupy_kernel<<<blocks, 32, smem, st>>>(ns, started);
  return (int)cudaGetLastError();
}
