// adam.cu -- standalone sharded mixed-precision Adam step.
//
// ("ZeRO-1/2/3", Stage 1 steps 5-6 and Stage 2: each rank updates the fp32
// optimizer state and master of its own shard with the reduced gradient, then
// writes the 16-bit parameter copy; "ZeRO Stage 2: Gradient Partitioning":
// the gradient shard is fp32 at the optimizer step.)
//
// Pure streaming: 16 bytes read + 14 bytes written per parameter (fp32 g,
// master, m, v in; master, m, v, bf16 param out).
#include "zpp_device.cuh"
#include "zpp_launch.h"

namespace zpp {
namespace {

constexpr int kAdamRows = 2;                          // 8-element vectors per lane per unit
constexpr int kAdamUnit = 32 * 8 * kAdamRows;         // 512 parameters per warp unit

struct AdamArgs {
  const float* g;
  float* master;
  float* m;
  float* v;
  uint16_t* param;
  int64_t n;
  AdamConsts ac;
};

__global__ void __launch_bounds__(kThreads) adam_kernel(const AdamArgs a) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int64_t units = (a.n + kAdamUnit - 1) / kAdamUnit;
  for (int64_t u = (int64_t)blockIdx.x * kWarps + warp; u < units;
       u += (int64_t)gridDim.x * kWarps) {
#pragma unroll
    for (int k = 0; k < kAdamRows; ++k) {
      const int64_t idx = u * kAdamUnit + (k * 32 + lane) * 8;
      if (idx + 8 <= a.n) {
        const float4* gp = reinterpret_cast<const float4*>(a.g + idx);
        const float4 g0 = __ldcs(gp), g1 = __ldcs(gp + 1);
        const float g[8] = {g0.x, g0.y, g0.z, g0.w, g1.x, g1.y, g1.z, g1.w};
        adam_update8(g, idx, a.master, a.m, a.v, a.param, a.ac);
      } else {
        for (int64_t i = idx; i < a.n; ++i) {
          float p = a.master[i], m = a.m[i], v = a.v[i];
          adam_update(a.g[i], p, m, v, a.ac);
          a.master[i] = p;
          a.m[i] = m;
          a.v[i] = v;
          if (a.param) a.param[i] = bf16_bits(p);
        }
      }
    }
  }
}

}  // namespace

cudaError_t launch_adam(const float* grad, int64_t n, const AdamConstsHost& ac, float* master,
                        float* m, float* v, uint16_t* param, cudaStream_t st) {
  AdamArgs a{grad, master, m, v, param, n,
             AdamConsts{ac.lr, ac.beta1, ac.beta2, ac.eps, ac.omb1, ac.omb2, ac.bc1, ac.bc2}};
  const int64_t units = (n + kAdamUnit - 1) / kAdamUnit;
  const void* k = reinterpret_cast<const void*>(&adam_kernel);
  adam_kernel<<<grid_for(k, (units + kWarps - 1) / kWarps), kThreads, 0, st>>>(a);
  return cudaGetLastError();
}

}  // namespace zpp
