// Exhaustive checks of device arithmetic identities the codec kernels rely on.
// Built and run by tests/test_gpu_device_identities.py on the GPU.
//
//  div_qmax<Q>(a) == __fdiv_rn(a, Q)   for every finite a >= 0, Q in {7, 127}
//  |recip(s) - __frcp_rn(s)| <= 1 ulp  for every s in [2^-100, 2^126)
#include <cstdio>
#include <cstdint>
#include <cuda_runtime.h>

#include "zpp_device.cuh"

__device__ unsigned long long g_bad[3];
__device__ unsigned int g_first[3];

__global__ void check(uint32_t lo, uint32_t hi) {
  const uint64_t stride = (uint64_t)gridDim.x * blockDim.x;
  for (uint64_t b = lo + (uint64_t)blockIdx.x * blockDim.x + threadIdx.x; b < hi; b += stride) {
    const float a = __uint_as_float((uint32_t)b);
    if (zpp::div_qmax<7>(a) != __fdiv_rn(a, 7.0f)) {
      if (atomicAdd(&g_bad[0], 1ull) == 0) g_first[0] = (uint32_t)b;
    }
    if (zpp::div_qmax<127>(a) != __fdiv_rn(a, 127.0f)) {
      if (atomicAdd(&g_bad[1], 1ull) == 0) g_first[1] = (uint32_t)b;
    }
    if (a >= zpp::kFastMinScale && a < zpp::kFastMaxScale) {
      const int d = (int)__float_as_uint(zpp::recip(a)) - (int)__float_as_uint(__frcp_rn(a));
      if (d > 1 || d < -1) {
        if (atomicAdd(&g_bad[2], 1ull) == 0) g_first[2] = (uint32_t)b;
      }
    }
  }
}

int main() {
  unsigned long long zero[3] = {0, 0, 0};
  if (cudaMemcpyToSymbol(g_bad, zero, sizeof zero) != cudaSuccess) return 2;
  int sms = 0;
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, 0);
  check<<<sms * 8, 256>>>(0u, 0x7F800000u);  // +0 .. largest finite
  if (cudaDeviceSynchronize() != cudaSuccess) return 3;
  unsigned long long bad[3];
  unsigned int first[3];
  cudaMemcpyFromSymbol(bad, g_bad, sizeof bad);
  cudaMemcpyFromSymbol(first, g_first, sizeof first);
  printf("div_qmax7 %llu %08x\n", bad[0], bad[0] ? first[0] : 0u);
  printf("div_qmax127 %llu %08x\n", bad[1], bad[1] ? first[1] : 0u);
  printf("recip_1ulp %llu %08x\n", bad[2], bad[2] ? first[2] : 0u);
  return 0;
}
