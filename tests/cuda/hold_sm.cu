// A kernel that holds SMs for a bounded time: each block takes enough shared
// memory that no verify CTA fits beside it, then sleeps until `cycles` of SM
// clock have passed.  Used to check that spec_verify finishes its work on the
// SMs it gets while other work holds the rest.
#include <cuda_runtime.h>

extern "C" __global__ void hold_sm(long long cycles, int* finished) {
  extern __shared__ unsigned char smem[];
  if (threadIdx.x == 0) smem[0] = 1;
  const long long t0 = clock64();
  while (clock64() - t0 < cycles) __nanosleep(1000);
  if (threadIdx.x == 0) atomicAdd(finished, 1);
}

extern "C" int launch_hold(int blocks, long long cycles, int smem_bytes, int* finished, void* stream) {
  cudaError_t e = cudaFuncSetAttribute(hold_sm, cudaFuncAttributeMaxDynamicSharedMemorySize, smem_bytes);
  if (e != cudaSuccess) return static_cast<int>(e);
  hold_sm<<<blocks, 128, smem_bytes, static_cast<cudaStream_t>(stream)>>>(cycles, finished);
  return static_cast<int>(cudaGetLastError());
}
