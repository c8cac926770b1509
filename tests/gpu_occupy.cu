// Test helper (not part of the library): a kernel that holds some SMs for a
// bounded time, so that a test can run a forward while only part of the GPU
// is free.  Each CTA takes enough dynamic shared memory that no second CTA of
// this kernel (and no CTA of the decode layer) fits beside it on its SM, and
// spins on the global timer until `ns` nanoseconds have passed; it always ends.
#include <cstdint>
#include <cuda_runtime.h>

__global__ void occupy_kernel(unsigned long long ns, int* done) {
  extern __shared__ int pad[];
  unsigned long long t0, t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t0));
  do {
    __nanosleep(1000);
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  } while (t - t0 < ns);
  if (threadIdx.x == 0) {
    pad[0] = 1;
    atomicAdd(done, pad[0]);
  }
}

extern "C" int occupy(int ctas, int smem_bytes, unsigned long long ns, int* done, void* stream) {
  if (ctas < 1 || smem_bytes < 1 || ns > 2000000000ull) return -1;   // at most 2 s
  cudaError_t e = cudaFuncSetAttribute(occupy_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem_bytes);
  if (e != cudaSuccess) return -2;
  occupy_kernel<<<ctas, 128, smem_bytes, static_cast<cudaStream_t>(stream)>>>(ns, done);
  return cudaGetLastError() == cudaSuccess ? 0 : -3;
}
