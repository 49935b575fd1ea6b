// Test helper: evaluates cuRAND's device Philox4x32-10 block function and the
// library's own Philox (csrc/philox.cuh) on the same counters and keys, so the
// tests can compare both with each other and with the CPU oracle.
#include <cuda_runtime.h>
#include <curand_kernel.h>
#include <stdint.h>

#include "philox.cuh"

__global__ void philox_pin_kernel(const uint4* ctr, const uint2* key, uint4* by_curand, uint4* by_lib,
                                  int n) {
  const int i = blockIdx.x * blockDim.x + threadIdx.x;
  if (i >= n) return;
  by_curand[i] = curand_Philox4x32_10(ctr[i], key[i]);
  const specdec::Philox4 r = specdec::philox4x32_10(ctr[i].x, ctr[i].y, ctr[i].z, ctr[i].w, key[i].x, key[i].y);
  by_lib[i] = make_uint4(r.w[0], r.w[1], r.w[2], r.w[3]);
}

__global__ void uniform_pin_kernel(const uint32_t* w, float* u, int n) {
  const int i = blockIdx.x * blockDim.x + threadIdx.x;
  if (i < n) u[i] = specdec::uniform_from_word(w[i]);
}

extern "C" int philox_pin(const void* ctr, const void* key, void* by_curand, void* by_lib, int n) {
  philox_pin_kernel<<<(n + 127) / 128, 128>>>(static_cast<const uint4*>(ctr), static_cast<const uint2*>(key),
                                               static_cast<uint4*>(by_curand), static_cast<uint4*>(by_lib), n);
  return static_cast<int>(cudaDeviceSynchronize());
}

extern "C" int uniform_pin(const void* w, void* u, int n) {
  uniform_pin_kernel<<<(n + 127) / 128, 128>>>(static_cast<const uint32_t*>(w), static_cast<float*>(u), n);
  return static_cast<int>(cudaDeviceSynchronize());
}
